// RoPE-mode decode attention with the key rebuild on tcgen05 tensor cores.
//
// "Palu: KV-Cache Compression With Low-Rank Projection", supplementary section
// (online-rebuild score kernel): the latent keys H (L x r) are streamed tile by
// tile, each tile is multiplied by the reconstruction matrix B on chip, RoPE is
// applied to the rebuilt keys and they are dotted with the query; intermediates
// never leave the chip. Here, per CTA:
//   * one (batch row b, group g, head pair hp, T-split) unit; the head pair's
//     slice of B_k^T (256 rows x r, K-major, the two heads' rows interleaved so a
//     dimension's two heads land in adjacent accumulator columns) stays in shared
//     memory;
//   * fp16 / int4 operands: the rotated query is folded into that slice once, so the
//     MMA yields q_a k_a + q_b k_b and q_b k_a - q_a k_b per rotation pair directly;
//     bf16 operands rebuild K exactly and apply the query in the epilogue;
//   * warp 0 streams 128-token x 64-rank chunks of H_k,g by TMA (128-byte swizzle)
//     through a 3-stage ring (int4: packed tiles, expanded to exact fp16 codes by a
//     converter warpgroup); warp 2 streams H_v,g chunks by TMA through a ring;
//   * warp 1 issues tcgen05.mma (M=128 tokens, N=256 = 2 heads x d_h, K=r) into
//     one of two TMEM accumulators;
//   * two score warpgroups (one token row per thread, read with tcgen05.ld; each
//     takes half of the 64 rotation pairs) apply the rotation at the token's position
//     with packed f32x2 FMAs for both heads, leaving partial scores of the tile in a
//     double-buffered slot in shared memory;
//   * two softmax warpgroups run the same online softmax (base 2) on the previous
//     tile's scores; for p H_v each lane owns 8 of the 256 value columns and the
//     warps share out the tokens (fp16/bf16: packed FMAs; int4: dp2a on the raw codes
//     with 15-bit weights), so scoring and p H_v of consecutive tiles overlap;
//   * the last CTA of a unit merges the T-split partials, so a decode is one launch;
//   * setmaxnreg moves registers from the control warpgroup to the score warpgroups.
// RoPE angles: pair k's frequency is held as a 64-bit fixed-point fraction of a
// turn F_k, so position p's phase is (p * F_k mod 2^64) / 2^64 turns: integer
// range reduction with no rounding (phase accumulation as in direct digital
// synthesis); the top 32 bits become an angle in [-pi, pi) for __sincosf.
// Every mbarrier wait is bounded; a time-out sets the workspace error word
// (PALU_ERR_TIMEOUT), all roles stop, in-flight copies are drained and TMEM freed.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "split_merge.cuh"
#include "tc_ptx.cuh"

namespace palu {

namespace {

constexpr int kTile = 128;                       // tokens per tile (MMA M)
constexpr int kHeads = 2;                        // heads per CTA
constexpr int kDh = 128;                         // head dim
constexpr int kHalf = kDh / 2;                   // RoPE pairs per head
constexpr int kN = kHeads * kDh;                 // MMA N
constexpr int kRank = 256;                       // r_k = r_v (MMA K)
constexpr int kKChunk = 64;                      // K elements per 128-byte swizzled row
constexpr int kChunks = kRank / kKChunk;         // 4
constexpr int kAStage = kTile * kKChunk * 2;     // 16 KB fp16 operand chunk
constexpr int kBChunk = kN * kKChunk * 2;        // 32 KB
constexpr int kBBytes = kBChunk * kChunks;       // 128 KB
constexpr int kWg = 128;                         // threads per warpgroup
constexpr uint32_t kTmemCols = 512;              // two N=256 fp32 accumulators

constexpr float kTurnToRad = 1.4629180792671596e-09f;  // 2 pi / 2^32

// Per-variant layout. I4K = int4 key latents: the H_k tile arrives packed (16 KB) and a converter
// warpgroup expands it into the fp16 operand ring. I4V = int4 value latents: H_v chunks hold
// packed rows (64 tokens each) for the dp2a p H_v.
// Warpgroups: 0 = warp 0 H_k/B producer, warp 1 MMA issuer, warp 2 H_v producer, warp 3 idle;
// 1, 2 = score warpgroups (rotation pairs 0-31 / 32-63); 3, 4 = softmax/PV warpgroups
// (value columns 0-127 / 128-255); 5 = int4 key converter (I4K only).
template <bool I4K, bool I4V>
struct Lay {
  static constexpr int kThreads = (I4K ? 6 : 5) * kWg;
  static constexpr int kLaunchRegs = I4K ? 80 : 96;  // per thread at launch (launch bounds, one CTA per SM)
  static constexpr int kRegsCtl = I4K ? 40 : 48, kRegsScore = I4K ? 128 : 152, kRegsPv = 64, kRegsConv = 48;
  static constexpr int kStages = I4K ? 2 : 3;        // fp16 H_k operand ring
  static constexpr int kPStages = I4K ? 2 : 0;       // packed int4 H_k tiles
  static constexpr int kPStage = kTile * (kRank / 2);
  // tokens per H_v chunk: 32-token fp16/bf16 chunks in two slots beat 16-token chunks in five
  // (bf16 B8 T32K: 651 vs 725 us on GB300): half the slot hand-offs per tile
  static constexpr int kVTok = I4V ? 64 : 32;
  static constexpr int kVRow = I4V ? kRank / 2 : kRank * 2;
  static constexpr int kVSlot = kVTok * kVRow;      // 8 KB (int4) or 16 KB (fp16 / bf16)
  static constexpr int kVSlots = I4V ? (I4K ? 2 : 4) : 2;
  static constexpr int kVChunks = kTile / kVTok;
  static constexpr int kOffB = 0;
  static constexpr int kOffA = kOffB + kBBytes;
  static constexpr int kOffPk = kOffA + kStages * kAStage;
  static constexpr int kOffV = kOffPk + kPStages * kPStage;
  static constexpr int kOffBar = kOffV + kVSlots * kVSlot;
  static constexpr int kNumBars = 52;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kOffQ = (kOffMisc + 16 + 15) & ~15;     // float4 [kHalf]: (qa0, qa1, qb0, qb1)
  static constexpr int kOffF = kOffQ + kHalf * 16;             // uint64 [kHalf]
  static constexpr int kOffS = kOffF + kHalf * 8;              // float2 [2 buf][2 part][kTile]
  static constexpr int kOffRed = kOffS + 4 * kTile * 8;        // float2 [2 wg][4]
  static constexpr int kOffP = kOffRed + 2 * 4 * 8;            // float2 [2 wg][kTile]
  static constexpr int kOffL = kOffP + 2 * kTile * 8;          // float2 [2 wg][4]
  static constexpr int kSmemBytes = kOffL + 2 * 4 * 8;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr int kOffO = kOffV;                          // [8 warps][kHeads][kRank] floats
  static_assert(kWg * kRegsCtl + 2 * kWg * kRegsScore + 2 * kWg * kRegsPv + (I4K ? kWg * kRegsConv : 0) <=
                    kThreads * kLaunchRegs,
                "register split");
  static_assert(8 * kHeads * kRank * 4 <= kVSlots * kVSlot, "output reduction fits the H_v ring");
  static_assert(kHeads * (256 + 2) * 4 <= kVSlots * kVSlot, "split-merge scratch fits the H_v ring");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

struct TcParams {
  DecodeArgs a;
  int hp_count;   // head pairs per group
  int bf16;       // MMA operand type
};

// d += a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) / b.byte2, b.byte3 (hi), unsigned
__device__ __forceinline__ uint32_t dp2a_lo(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp2a.lo.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp2a_hi(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp2a.hi.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// eight fp16 / bf16 values (16 bytes) as four float pairs
__device__ __forceinline__ void vt8_to_float2x4(const uint4& u, float2* f, __half) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
}
__device__ __forceinline__ void vt8_to_float2x4(const uint4& u, float2* f, __nv_bfloat16) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
}

// eight signed 4-bit codes of a 32-bit word (element 2j = low nibble of byte j) as eight
// exact fp16 values, in the order [0, 2, 4, 6, 1, 3, 5, 7] (B_k^T is stored with its ranks
// permuted alike): each nibble biased by 8 is placed under the fp16 exponent of 1024 (0x64xx),
// and 1032 is subtracted.
__device__ __forceinline__ uint4 int4x8_to_half8(uint32_t w) {
  const uint32_t lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u;          // elements 0, 2, 4, 6
  const uint32_t hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // elements 1, 3, 5, 7
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
  uint32_t r[4];
  r[0] = __byte_perm(lo, 0x64646464u, 0x4140);
  r[1] = __byte_perm(lo, 0x64646464u, 0x4342);
  r[2] = __byte_perm(hi, 0x64646464u, 0x4140);
  r[3] = __byte_perm(hi, 0x64646464u, 0x4342);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&r[i]), bias);
    r[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// The int4 key converter's work on one token row and one 64-rank chunk: packed bytes
// 32 kc .. 32 kc + 31 of the row (16-byte chunks 2 kc and 2 kc + 1 of a tile loaded by TMA with
// the 128-byte swizzle, row r) become 64 exact fp16 codes, written as row r of the 128-byte-
// swizzled fp16 MMA operand chunk `arow` points into (arow = chunk base + 128 r).
__device__ __forceinline__ void convert_int4_row_chunk(const uint8_t* prow, uint8_t* arow, int r, int kc) {
  const uint4 w0 = *reinterpret_cast<const uint4*>(prow + (((2 * kc) ^ (r & 7)) << 4));
  const uint4 w1 = *reinterpret_cast<const uint4*>(prow + (((2 * kc + 1) ^ (r & 7)) << 4));
  const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(arow + ((j ^ (r & 7)) << 4)) = int4x8_to_half8(wv[j]);
}

// int4 p H_v on the raw value codes, per warp: 16 tokens (two groups of eight, ch = 0, 1) and two
// heads. Lane l holds the 15-bit integer weight q of token l & 15 (group (l & 15) >> 3) for head
// l >> 4; dp2a_pack_weights pairs neighbouring tokens' weights (valid in even lanes) and sums the
// warp's weights per head.
__device__ __forceinline__ void dp2a_pack_weights(uint32_t qv, uint32_t& qpair, uint32_t& qsum) {
  qsum = qv;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
  qpair = qv | (__shfl_down_sync(0xffffffffu, qv, 1) << 16);
}

// Accumulate sum_k q_k (code_k + 8) over the eight tokens of group ch for this lane's eight value
// columns (8 lane .. 8 lane + 7) and both heads, exactly in int32. u[k] = the lane's four packed
// bytes of token k of the group. dp2a multiplies two tokens' 16-bit weights by the two tokens'
// biased codes of one column (one byte each).
__device__ __forceinline__ void dp2a_accumulate8(const uint32_t (&u)[8], uint32_t qpair, int ch,
                                                 uint32_t (&ai)[2][8]) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t a0 = __shfl_sync(0xffffffffu, qpair, ch * 8 + 2 * m);
    const uint32_t a1 = __shfl_sync(0xffffffffu, qpair, 16 + ch * 8 + 2 * m);
    const uint32_t la = (u[2 * m] ^ 0x88888888u) & 0x0F0F0F0Fu;
    const uint32_t lb = (u[2 * m + 1] ^ 0x88888888u) & 0x0F0F0F0Fu;
    const uint32_t ha = ((u[2 * m] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    const uint32_t hb = ((u[2 * m + 1] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    const uint32_t b02 = __byte_perm(la, lb, 0x5140), b46 = __byte_perm(la, lb, 0x7362);
    const uint32_t b13 = __byte_perm(ha, hb, 0x5140), b57 = __byte_perm(ha, hb, 0x7362);
    ai[0][0] = dp2a_lo(a0, b02, ai[0][0]);
    ai[0][2] = dp2a_hi(a0, b02, ai[0][2]);
    ai[0][4] = dp2a_lo(a0, b46, ai[0][4]);
    ai[0][6] = dp2a_hi(a0, b46, ai[0][6]);
    ai[0][1] = dp2a_lo(a0, b13, ai[0][1]);
    ai[0][3] = dp2a_hi(a0, b13, ai[0][3]);
    ai[0][5] = dp2a_lo(a0, b57, ai[0][5]);
    ai[0][7] = dp2a_hi(a0, b57, ai[0][7]);
    ai[1][0] = dp2a_lo(a1, b02, ai[1][0]);
    ai[1][2] = dp2a_hi(a1, b02, ai[1][2]);
    ai[1][4] = dp2a_lo(a1, b46, ai[1][4]);
    ai[1][6] = dp2a_hi(a1, b46, ai[1][6]);
    ai[1][1] = dp2a_lo(a1, b13, ai[1][1]);
    ai[1][3] = dp2a_hi(a1, b13, ai[1][3]);
    ai[1][5] = dp2a_lo(a1, b57, ai[1][5]);
    ai[1][7] = dp2a_hi(a1, b57, ai[1][7]);
  }
}

// sum q code = sum q (code + 8) - 8 sum q, exact in int32 (|.| < 2^22)
__device__ __forceinline__ int32_t dp2a_unbias(uint32_t acc, uint32_t qsum_head) {
  return int32_t(acc - 8u * qsum_head);
}

// Fold the rotated query into B_k^T, in place, before the first MMA. B_k^T holds the head pair
// interleaved (row 2 d + j = dimension d of head j). For head j and rotation pair k, rows
// a = 2 k + j (dimension k) and b = a + 128 (dimension k + 64) become
//   U = q_a B_a + q_b B_b   and   W = q_b B_a - q_a B_b,
// so the MMA yields X_k = q_a k_a + q_b k_b and Y_k = q_b k_a - q_a k_b per token and the
// rotated score is sum_k cos X_k + sin Y_k. Rows a and b share their swizzle phase (a = b mod 8),
// so element m of both rows sits at the same offset in its row. Run by the 512 threads of the
// score and softmax warpgroups (tf = 0..511), one 64-column chunk at a time as its TMA lands;
// returns false if a wait gave up.
__device__ __forceinline__ bool fold_b(uint8_t* b_smem, const float4* qs, uint64_t* bfull, uint64_t* bready, int tf,
                                       int lane, volatile int* abort_flag, uint64_t wait_ns) {
  bool ok = true;
  for (int kc = 0; kc < kChunks; ++kc) {
    if (ok && !tc::mbar_wait_bounded(&bfull[kc], 0, abort_flag, wait_ns)) ok = false;
    if (ok) {
      uint8_t* chunk = b_smem + kc * kBChunk;
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int job = tf + rep * 4 * kWg;            // 0..1023: (head, pair, 16-byte chunk)
        const int c = job & 7, k = (job >> 3) & (kHalf - 1), j = job >> 9;
        const int ra = 2 * k + j;
        const float4 q4 = qs[k];
        const float qa = j ? q4.y : q4.x, qb = j ? q4.w : q4.z;
        uint4* pa = reinterpret_cast<uint4*>(chunk + ra * 128 + ((c ^ (ra & 7)) << 4));
        uint4* pb = reinterpret_cast<uint4*>(chunk + (ra + kDh) * 128 + ((c ^ (ra & 7)) << 4));
        uint4 va = *pa, vb = *pb;
        __half2* ha = reinterpret_cast<__half2*>(&va);
        __half2* hb = reinterpret_cast<__half2*>(&vb);
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const float2 ba = __half22float2(ha[e2]), bb = __half22float2(hb[e2]);
          const float2 uu = make_float2(fmaf(qa, ba.x, qb * bb.x), fmaf(qa, ba.y, qb * bb.y));
          const float2 ww = make_float2(fmaf(qb, ba.x, -qa * bb.x), fmaf(qb, ba.y, -qa * bb.y));
          ha[e2] = __float22half2_rn(uu);
          hb[e2] = __float22half2_rn(ww);
        }
        *pa = va;
        *pb = vb;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bready[kc]);
  }
  return ok;
}

__device__ __forceinline__ int token_position(const DecodeArgs& a, int b, int t, bool valid) {
  int pos = t;
  if (valid && a.positions) pos = a.positions[(int64_t)b * a.capacity + t];
  if (pos < 0 || pos >= a.max_pos) {
    if (valid) record_error(a.err, kCodeDevice, kErrPosition, pos, b);
    pos = pos < 0 ? 0 : int(a.max_pos - 1);
  }
  return pos;
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// VT = value-latent storage (__half, __nv_bfloat16, or Int4); I4K = int4 key latents (fp16 MMA operands);
// FOLD = the rotated query is folded into the B operand (fp16 operands only, see below)
template <typename VT, bool I4K, bool FOLD>
__global__ void __launch_bounds__(Lay<I4K, std::is_same<VT, Int4>::value>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_hk, const __grid_constant__ CUtensorMap tm_hv,
                     const __grid_constant__ CUtensorMap tm_b, const TcParams P) {
  constexpr bool I4V = std::is_same<VT, Int4>::value;   // int4 value latents (dp2a p H_v)
  using LY = Lay<I4K, I4V>;
  constexpr int kStages = LY::kStages, kPStages = LY::kPStages, kVSlots = LY::kVSlots, kVTok = LY::kVTok;
  constexpr int kVChunks = LY::kVChunks, kVSlot = LY::kVSlot, kVRow = LY::kVRow;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DecodeArgs& a = P.a;
  const uint64_t kWaitNs = a.wait_ns;   // bound of every mbarrier wait (1 s; shorter in the stall test)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = threadIdx.x / kWg;
  const int hp = blockIdx.x % P.hp_count, split = blockIdx.x / P.hp_count;
  const int g = blockIdx.y, b = blockIdx.z;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kOffBar);
  uint64_t* fullA = bars;                 // [kStages]
  uint64_t* emptyA = bars + 4;            // [kStages]
  uint64_t* bfull = bars + 8;             // [kChunks]
  uint64_t* tfull = bars + 12;            // [2]
  uint64_t* tempty = bars + 14;           // [2]
  uint64_t* vfull = bars + 16;            // [kVSlots]
  uint64_t* vempty = bars + 24;           // [kVSlots]
  uint64_t* sready = bars + 32;           // [2]
  uint64_t* sfree = bars + 34;            // [2]
  uint64_t* pfull = bars + 36;            // [kPStages]
  uint64_t* pempty = bars + 40;           // [kPStages]
  uint64_t* mma_done = bars + 44;
  uint64_t* bready = bars + 45;           // [kChunks] B chunk folded (FOLD only)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::kOffMisc + 4);
  float4* qs = reinterpret_cast<float4*>(smem + LY::kOffQ);
  uint64_t* Fs = reinterpret_cast<uint64_t*>(smem + LY::kOffF);
  float2* sbuf = reinterpret_cast<float2*>(smem + LY::kOffS);

  // this CTA's token range
  int T = a.seq_lens[b];
  if (T < 0 || T > a.max_seq_len) {
    if (threadIdx.x == 0 && split == 0 && hp == 0 && g == 0) record_error(a.err, kCodeDevice, kErrSeqLen, T, b);
    T = T < 0 ? 0 : a.max_seq_len;
  }
  const int span = a.tiles_per_split * kTile;
  const int t_begin = split * span;
  const int t_end = min(T, t_begin + span);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  const int head0 = g * a.s + hp * kHeads;  // first head of this CTA within the row
  const int row0 = b * (int)a.capacity;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&fullA[i], I4K ? 4 : 1);   // converter warps, or the TMA
      tc::mbar_init(&emptyA[i], 1);
    }
    for (int i = 0; i < kChunks; ++i) tc::mbar_init(&bfull[i], 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 8);   // lane 0 of the eight score warps
      tc::mbar_init(&sready[i], 8);   // eight score warps
      tc::mbar_init(&sfree[i], 8);    // eight softmax/PV warps
    }
    for (int i = 0; i < kVSlots; ++i) {
      tc::mbar_init(&vfull[i], 1);
      tc::mbar_init(&vempty[i], 8);   // eight softmax/PV warps
    }
    for (int i = 0; i < kPStages; ++i) {
      tc::mbar_init(&pfull[i], 1);
      tc::mbar_init(&pempty[i], 4);   // converter warps
    }
    tc::mbar_init(mma_done, 1);
    for (int i = 0; i < kChunks; ++i) tc::mbar_init(&bready[i], 16);  // score + softmax/PV warps
    *abort_flag = 0;
    tc::fence_barrier_init();
    if (n_tiles > 0) {
      // start B_k^T and the first operand tiles now, so their latency overlaps the query
      // rotation and the TMEM allocation (this thread is the producer; the rings are empty)
      tc::tma_prefetch(&tm_hk);
      tc::tma_prefetch(&tm_b);
      const int brow = g * (a.s * kDh) + hp * kN;
      for (int kc = 0; kc < kChunks; ++kc) {
        tc::mbar_arrive_expect_tx(&bfull[kc], kBChunk);
        tc::tma_load_2d(smem + LY::kOffB + kc * kBChunk, &tm_b, &bfull[kc], kc * kKChunk, brow);
      }
      if constexpr (I4K) {
        for (int it = 0; it < min(kPStages, n_tiles); ++it) {
          tc::mbar_arrive_expect_tx(&pfull[it], LY::kPStage);
          tc::tma_load_3d(smem + LY::kOffPk + it * LY::kPStage, &tm_hk, &pfull[it], 0, g, row0 + t_begin + it * kTile);
        }
      } else {
        for (int ci = 0; ci < min(kStages, kChunks * n_tiles); ++ci) {
          tc::mbar_arrive_expect_tx(&fullA[ci], kAStage);
          tc::tma_load_3d(smem + LY::kOffA + ci * kAStage, &tm_hk, &fullA[ci], (ci % kChunks) * kKChunk, g,
                          row0 + t_begin + (ci / kChunks) * kTile);
        }
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (wg == 1) {
    // rotate the two heads' queries at q_pos (RoPE table, float64-derived), scale by
    // log2(e)/sqrt(d_h), and keep them as (q_a, q_b) pairs per rotation pair
    const int i = threadIdx.x - kWg;
    const int j = i / kHalf, k = i % kHalf;
    int qp = 0;
    if (a.q_pos) qp = a.q_pos[b];
    else if (T > 0) qp = a.positions ? a.positions[(int64_t)b * a.capacity + (T - 1)] : (T - 1);
    if (qp < 0 || qp >= a.max_pos) {
      if (i == 0 && split == 0 && hp == 0 && g == 0) record_error(a.err, kCodeDevice, kErrQueryPos, qp, b);
      qp = qp < 0 ? 0 : int(a.max_pos - 1);
    }
    const float2 cs = a.rope[(int64_t)qp * kHalf + k];
    const int64_t qoff = ((int64_t)b * a.n_heads + head0 + j) * kDh;
    const float x0 = load_as_f32(a.q, a.q_dtype, qoff + k);
    const float x1 = load_as_f32(a.q, a.q_dtype, qoff + k + kHalf);
    float* qf = reinterpret_cast<float*>(&qs[k]);
    qf[j] = (x0 * cs.x - x1 * cs.y) * a.qscale;
    qf[2 + j] = (x1 * cs.x + x0 * cs.y) * a.qscale;
    if (j == 0) Fs[k] = a.phase[k];
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (wg == 0) {
    setmaxnreg_dec<LY::kRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- H_k / B producer
      if (lane == 0 && n_tiles > 0) {
        // B_k^T and the first ring fills were issued in the prologue
        bool ok = true;
        if constexpr (I4K) {
          // whole packed tiles (128 tokens x 128 bytes) into the staging ring
          int issued = min(kPStages, n_tiles);
          for (int it = issued; it < n_tiles && ok; ++it) {
            const int ps = it % kPStages;
            if (!tc::mbar_wait_bounded(&pempty[ps], ((it / kPStages) & 1) ^ 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc::mbar_arrive_expect_tx(&pfull[ps], LY::kPStage);
            tc::tma_load_3d(smem + LY::kOffPk + ps * LY::kPStage, &tm_hk, &pfull[ps], 0, g, row0 + t_begin + it * kTile);
            ++issued;
          }
          if (!ok) {
            volatile int quiet = 0;
            for (int it = (issued > kPStages ? issued - kPStages : 0); it < issued; ++it)
              tc::mbar_wait_bounded(&pfull[it % kPStages], (it / kPStages) & 1, &quiet, kWaitNs / 10);
          }
        } else {
          // operand chunk ci = (tile ci / 4, 64-column chunk ci % 4) goes to stage ci % kStages
          int issued = min(kStages, kChunks * n_tiles);
          for (int ci = issued; ci < kChunks * n_tiles && ok; ++ci) {
            const int stage = ci % kStages;
            const uint32_t round = uint32_t(ci / kStages);
            if (!tc::mbar_wait_bounded(&emptyA[stage], (round & 1) ^ 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc::mbar_arrive_expect_tx(&fullA[stage], kAStage);
            tc::tma_load_3d(smem + LY::kOffA + stage * kAStage, &tm_hk, &fullA[stage], (ci % kChunks) * kKChunk, g,
                            row0 + t_begin + (ci / kChunks) * kTile);
            ++issued;
          }
          if (!ok) {
            // drain the copies still in flight before the CTA may exit
            volatile int quiet = 0;
            for (int ci = (issued > kStages ? issued - kStages : 0); ci < issued; ++ci)
              tc::mbar_wait_bounded(&fullA[ci % kStages], uint32_t(ci / kStages) & 1, &quiet, kWaitNs / 10);
          }
        }
        if (!ok) {
          volatile int quiet = 0;
          for (int kc = 0; kc < kChunks; ++kc) tc::mbar_wait_bounded(&bfull[kc], 0, &quiet, kWaitNs / 10);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && n_tiles > 0) {
        const uint32_t idesc = tc::idesc_f16(kTile, kN, P.bf16 != 0);
        bool ok = true;
        int stage = 0;
        uint32_t round = 0;
        const uint32_t a_base = tc::smem_addr(smem + LY::kOffA);
        const uint32_t b_base = tc::smem_addr(smem + LY::kOffB);
        for (int it = 0; it < n_tiles && ok; ++it) {
          const int buf = it & 1;
          const uint32_t use = it >> 1;
          if (!tc::mbar_wait_bounded(&tempty[buf], (use & 1) ^ 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t d = tmem_base + buf * kN;
          for (int kc = 0; kc < kChunks; ++kc) {
            if (it == 0 && !tc::mbar_wait_bounded(FOLD ? &bready[kc] : &bfull[kc], 0, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            if (!tc::mbar_wait_bounded(&fullA[stage], round & 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < kKChunk / 16; ++k) {
              const uint64_t ad = tc::sdesc_k_sw128(a_base + stage * kAStage + k * 32);
              const uint64_t bd = tc::sdesc_k_sw128(b_base + kc * kBChunk + k * 32);
              tc::umma_f16(d, ad, bd, idesc, (kc | k) != 0);
            }
            tc::umma_commit(&emptyA[stage]);
            if (++stage == kStages) {
              stage = 0;
              ++round;
            }
          }
          if (!ok) break;
          tc::umma_commit(&tfull[buf]);
        }
        // every MMA this thread issued has completed once mma_done flips
        tc::umma_commit(mma_done);
        volatile int quiet = 0;
        tc::mbar_wait_bounded(mma_done, 0, &quiet, kWaitNs);
      }
    } else if (warp == 2) {
      // ---------------------------------------------------------- H_v producer
      if (lane == 0 && n_tiles > 0 && !a.test_stall) {
        tc::tma_prefetch(&tm_hv);
        int issued = 0;
        bool ok = true;
        for (int it = 0; it < n_tiles && ok; ++it) {
          const int t0 = t_begin + it * kTile;
          for (int ch = 0; ch < kVChunks; ++ch) {
            const int vi = it * kVChunks + ch;
            const int slot = vi % kVSlots;
            if (!tc::mbar_wait_bounded(&vempty[slot], ((vi / kVSlots) & 1) ^ 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc::mbar_arrive_expect_tx(&vfull[slot], kVSlot);
            tc::tma_load_3d(smem + LY::kOffV + slot * kVSlot, &tm_hv, &vfull[slot], 0, g, row0 + t0 + ch * kVTok);
            ++issued;
          }
        }
        if (!ok) {
          volatile int quiet = 0;
          for (int vi = (issued > kVSlots ? issued - kVSlots : 0); vi < issued; ++vi)
            tc::mbar_wait_bounded(&vfull[vi % kVSlots], (vi / kVSlots) & 1, &quiet, kWaitNs / 10);
        }
      }
    }
  } else if (wg <= 2) {
    // ------------------------------------------------------------ score warpgroups
    // thread = one token row of the tile; warpgroup X handles rotation pairs 32X..32X+31 of
    // both heads: rotate each rebuilt key pair at the token's position, dot it with the
    // rotated query, and leave the partial scores in shared memory. For int4 latents the MMA
    // ran on the integer codes and the token's key scale multiplies the score (RoPE and the
    // dot product are linear in the key).
    setmaxnreg_inc<LY::kRegsScore>();
    if (FOLD && n_tiles > 0) fold_b(smem + LY::kOffB, qs, bfull, bready, threadIdx.x - kWg, lane, abort_flag, kWaitNs);
    const int X = wg - 1;
    const int quad = warp & 3;               // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    bool slot_lost = false;   // warp-uniform: a score-slot wait gave up
    int pos_next = token_position(a, b, t_begin + row, t_begin + row < t_end);
    float ks_next = 1.f;
    if constexpr (I4K)
      if (t_begin + row < t_end) ks_next = __half2float(a.k_scale[((int64_t)row0 + t_begin + row) * a.n_g + g]);
    for (int it = 0; it < n_tiles; ++it) {
      const int buf = it & 1;
      const uint32_t use = it >> 1;
      const int t0 = t_begin + it * kTile;
      const bool valid = t0 + row < t_end;
      const uint32_t upos = uint32_t(pos_next);
      const float ks = ks_next;
      if (it + 1 < n_tiles) {
        const int tn = t0 + kTile + row;
        pos_next = token_position(a, b, tn, tn < t_end);
        if constexpr (I4K)
          if (tn < t_end) ks_next = __half2float(a.k_scale[((int64_t)row0 + tn) * a.n_g + g]);
      }

      // the score slot is needed only for the final write: wait for the accumulator now and
      // for the slot after the math, so TMEM goes back to the MMA as early as possible
      const bool got = tc::mbar_wait_bounded(&tfull[buf], use & 1, abort_flag, kWaitNs);
      if (tc::named_bar_or(1 + X, kWg, !got || slot_lost)) break;  // one decision for the warpgroup
      tc::tc_fence_after();

      // accumulator columns: 2 d + j = dimension d of head j, so (head 0, head 1) of a dimension
      // are adjacent and one packed f32x2 instruction updates both heads
      float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
      const uint32_t tbase = tmem_base + (uint32_t(quad * 32) << 16) + buf * kN;
#pragma unroll 1
      for (int a0 = 32 * X; a0 < 32 * X + 32; a0 += 16) {
        // issue the four TMEM loads of this chunk (dimensions a0..a0+15 and a0+64..a0+79 of
        // both heads), compute the chunk's cos/sin while they are in flight, then wait
        uint32_t ka[32], kb[32];
        tc::tmem_ld16x2_nowait(tbase + 2 * a0, tbase + 2 * a0 + 16, ka);
        tc::tmem_ld16x2_nowait(tbase + kDh + 2 * a0, tbase + kDh + 2 * a0 + 16, kb);
        float cs[16], sn[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint64_t F = Fs[a0 + u];
          const uint32_t top = __umulhi(upos, uint32_t(F)) + upos * uint32_t(F >> 32);
          __sincosf(float(int32_t(top)) * kTurnToRad, &sn[u], &cs[u]);
        }
        tc::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 c2 = make_float2(cs[u], cs[u]), s2 = make_float2(sn[u], sn[u]);
          const float2 xa = make_float2(__uint_as_float(ka[2 * u]), __uint_as_float(ka[2 * u + 1]));
          const float2 xb = make_float2(__uint_as_float(kb[2 * u]), __uint_as_float(kb[2 * u + 1]));
          float2& acc = (u & 1) ? sb : sa;
          if constexpr (FOLD) {
            // the MMA produced X_k (xa) and Y_k (xb) directly
            acc = __ffma2_rn(c2, xa, acc);
            acc = __ffma2_rn(s2, xb, acc);
          } else {
            // c (q_a k_a + q_b k_b) + s (q_b k_a - q_a k_b) = k_a (c q_a + s q_b) + k_b (c q_b - s q_a)
            const float4 q4 = qs[a0 + u];     // (qa0, qa1, qb0, qb1)
            const float2 qa = make_float2(q4.x, q4.y), qb = make_float2(q4.z, q4.w);
            const float2 al = __ffma2_rn(s2, qb, __fmul2_rn(c2, qa));
            const float2 be = __ffma2_rn(make_float2(-sn[u], -sn[u]), qa, __fmul2_rn(c2, qb));
            acc = __ffma2_rn(xa, al, acc);
            acc = __ffma2_rn(xb, be, acc);
          }
        }
      }
      const float s0a = sa.x, s0b = sb.x, s1a = sa.y, s1b = sb.y;
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);
      // a slot wait that gave up skips the write; the next tile's barrier-OR ends the loop
      slot_lost = __any_sync(0xffffffffu, !tc::mbar_wait_bounded(&sfree[buf], (use & 1) ^ 1, abort_flag, kWaitNs));
      if (!slot_lost) {
        sbuf[(buf * 2 + X) * kTile + row] =
            valid ? make_float2((s0a + s0b) * ks, (s1a + s1b) * ks) : make_float2(-INFINITY, -INFINITY);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sready[buf]);
      }
    }
  } else if (wg <= 4) {
    // ------------------------------------------------------------ softmax / PV warpgroups
    // Both warpgroups run the same online softmax over the tile's 128 scores (summing the two
    // partial scores). For p H_v every lane owns 8 of the 256 value columns (lane 8 .. lane 8 + 7)
    // and the eight warps share out each H_v chunk's tokens; packed f32x2 FMAs update both
    // heads' column pairs. For int4 latents p is multiplied by the token's value scale before
    // it weights the codes.
    setmaxnreg_dec<LY::kRegsPv>();
    const int Y = wg - 3;
    const int e = warp & 3;                  // warp within the warpgroup
    const int ei = threadIdx.x - wg * kWg;   // 0..127: token row for the softmax
    const int bar = 3 + Y;
    float2* red = reinterpret_cast<float2*>(smem + LY::kOffRed) + Y * 4;
    float2* pbuf = reinterpret_cast<float2*>(smem + LY::kOffP) + Y * kTile;
    float2* lred = reinterpret_cast<float2*>(smem + LY::kOffL) + Y * 4;
    float* ored = reinterpret_cast<float*>(smem + LY::kOffO);  // [8 warps][kHeads][kRank] at the end
    const int w8 = Y * 4 + e;                                   // warp among the eight
    float m_run0 = -INFINITY, m_run1 = -INFINITY;
    float l0 = 0.f, l1 = 0.f;
    float2 acc0[4], acc1[4];     // columns (lane 8 + 2 j, lane 8 + 2 j + 1) of head 0 / head 1
#pragma unroll
    for (int c = 0; c < 4; ++c) acc0[c] = acc1[c] = make_float2(0.f, 0.f);
    bool aborted = false;  // warpgroup-uniform: only ever set from a barrier-OR
    bool broken = false;   // this warp's own H_v wait gave up
    if (FOLD && n_tiles > 0) {  // (B_k is loaded only when the CTA has tokens)
      if (!fold_b(smem + LY::kOffB, qs, bfull, bready, threadIdx.x - kWg, lane, abort_flag, kWaitNs)) broken = true;
    }
    float vs_next = 1.f;
    if constexpr (I4V)
      if (t_begin + ei < t_end) vs_next = __half2float(a.v_scale[((int64_t)row0 + t_begin + ei) * a.n_g + g]);

    for (int it = 0; it < n_tiles; ++it) {
      const int buf = it & 1;
      const uint32_t use = it >> 1;
      const int t0 = t_begin + it * kTile;
      const float vsc = vs_next;
      if constexpr (I4V)
        if (it + 1 < n_tiles && t0 + kTile + ei < t_end)
          vs_next = __half2float(a.v_scale[((int64_t)row0 + t0 + kTile + ei) * a.n_g + g]);
      const bool got = tc::mbar_wait_bounded(&sready[buf], use & 1, abort_flag, kWaitNs);
      if (tc::named_bar_or(bar, kWg, !got || broken)) {
        aborted = true;
        break;
      }
      const float2 pa = sbuf[(buf * 2 + 0) * kTile + ei];
      const float2 pb = sbuf[(buf * 2 + 1) * kTile + ei];
      const float2 sc = make_float2(pa.x + pb.x, pa.y + pb.y);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sfree[buf]);

      // online softmax over the tile (uniform running max across the 128 threads)
      const float w0 = warp_max(sc.x), w1 = warp_max(sc.y);
      if (lane == 0) red[e] = make_float2(w0, w1);
      tc::named_bar(bar, kWg);
      float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tm0 = fmaxf(tm0, red[k].x);
        tm1 = fmaxf(tm1, red[k].y);
      }
      const float mn0 = fmaxf(m_run0, tm0), mn1 = fmaxf(m_run1, tm1);
      const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m_run0 - mn0);
      const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m_run1 - mn1);
      const float p0 = (sc.x == -INFINITY) ? 0.f : exp2f(sc.x - mn0);
      const float p1 = (sc.y == -INFINITY) ? 0.f : exp2f(sc.y - mn1);
      m_run0 = mn0;
      m_run1 = mn1;
      l0 = l0 * al0 + p0;
      l1 = l1 * al1 + p1;
      pbuf[ei] = I4V ? make_float2(p0 * vsc, p1 * vsc) : make_float2(p0, p1);
      tc::named_bar(bar, kWg);

      {
        const float2 a0 = make_float2(al0, al0), a1 = make_float2(al1, al1);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc0[c] = __fmul2_rn(acc0[c], a0);
          acc1[c] = __fmul2_rn(acc1[c], a1);
        }
      }
      if constexpr (I4V) {
        // p H_v on the integer codes. Warp w8 owns tokens 64 ch + 8 w8 .. 64 ch + 8 w8 + 7 of
        // chunks ch = 0, 1 (16 tokens); lane l quantises the weight p' = p * v_scale of token
        // (l & 15) for head l >> 4 to 15 bits against the largest of the warp's 16 weights of that
        // head, q = rint(p' * 32767 / S). Then dp2a multiplies two tokens' weights by their biased
        // codes (code + 8, bytes) per column, with exact int32 sums; subtracting 8 * sum(q) removes
        // the bias. The rounding of q errs by at most S / 65534 per weight.
        const int jt = lane & 15, hh = lane >> 4;
        const int tkq = (jt >> 3) * kVTok + w8 * 8 + (jt & 7);
        const float2 pq = pbuf[tkq];
        const float pw = hh ? pq.y : pq.x;
        float smax = pw;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        const float inv = smax > 0.f ? 32767.f / smax : 0.f;
        const uint32_t qv = uint32_t(__float2int_rn(pw * inv));
        uint32_t qsum, qpair;
        dp2a_pack_weights(qv, qpair, qsum);
        uint32_t ai[2][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) ai[0][c] = ai[1][c] = 0u;
        for (int ch = 0; ch < kVChunks; ++ch) {
          const int vi = it * kVChunks + ch;
          const int slot = vi % kVSlots;
          if (!tc::mbar_wait_bounded(&vfull[slot], (vi / kVSlots) & 1, abort_flag, kWaitNs)) broken = true;
          broken = __any_sync(0xffffffffu, broken);   // warp-uniform before the shuffles below
          const uint8_t* vs = smem + LY::kOffV + slot * kVSlot + (w8 * 8) * kVRow + lane * 4;
          uint32_t u[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) u[k] = *reinterpret_cast<const uint32_t*>(vs + k * kVRow);
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&vempty[slot]);
          if (broken) continue;
          dp2a_accumulate8(u, qpair, ch, ai);
        }
        if (!broken) {
          // back to float: sum(q * code) = sum(q * (code + 8)) - 8 sum(q), |.| < 2^22
          const uint32_t qs0 = __shfl_sync(0xffffffffu, qsum, 0), qs1 = __shfl_sync(0xffffffffu, qsum, 16);
          const float sc0 = __shfl_sync(0xffffffffu, smax, 0) * (1.f / 32767.f);
          const float sc1 = __shfl_sync(0xffffffffu, smax, 16) * (1.f / 32767.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float2 v0 = make_float2(float(dp2a_unbias(ai[0][2 * c], qs0)), float(dp2a_unbias(ai[0][2 * c + 1], qs0)));
            const float2 v1 = make_float2(float(dp2a_unbias(ai[1][2 * c], qs1)), float(dp2a_unbias(ai[1][2 * c + 1], qs1)));
            acc0[c] = __ffma2_rn(v0, make_float2(sc0, sc0), acc0[c]);
            acc1[c] = __ffma2_rn(v1, make_float2(sc1, sc1), acc1[c]);
          }
        }
      } else {
        // p H_v on fp16/bf16 rows: chunk ch of the tile holds kVTok = 32 tokens and warp w8 takes
        // four of them. A warp whose wait gave up skips the arithmetic; the tile-level barrier-OR
        // above then ends the loop for the warpgroup.
        constexpr int kPer = kVTok / 8;
        for (int ch = 0; ch < kVChunks; ++ch) {
          const int vi = it * kVChunks + ch;
          const int slot = vi % kVSlots;
          if (!tc::mbar_wait_bounded(&vfull[slot], (vi / kVSlots) & 1, abort_flag, kWaitNs)) broken = true;
          const uint8_t* vs = smem + LY::kOffV + slot * kVSlot + (w8 * kPer) * kVRow;
          uint4 u[kPer];
#pragma unroll
          for (int k = 0; k < kPer; ++k) u[k] = *reinterpret_cast<const uint4*>(vs + k * kVRow + lane * 16);
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&vempty[slot]);
          if (broken) continue;
          const int tk0 = ch * kVTok + w8 * kPer;   // first token (within the tile) of this warp
          const bool all = t0 + tk0 + kPer - 1 < t_end;
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            if (all || t0 + tk0 + k < t_end) {
              float2 h[4];
              vt8_to_float2x4(u[k], h, VT{});
              const float2 p = pbuf[tk0 + k];
              const float2 p0 = make_float2(p.x, p.x), p1 = make_float2(p.y, p.y);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                acc0[c] = __ffma2_rn(p0, h[c], acc0[c]);
                acc1[c] = __ffma2_rn(p1, h[c], acc1[c]);
              }
            }
          }
        }
      }
    }

    // reduce the eight warps' partial sums and write this split's partials; the decision is
    // taken over both warpgroups at once, so either both or neither enter the barriers below
    aborted = tc::named_bar_or(7, 2 * kWg, aborted || broken || *abort_flag != 0);
    if (!aborted) {
      const float ls0 = warp_sum(l0), ls1 = warp_sum(l1);
      if (lane == 0) lred[e] = make_float2(ls0, ls1);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        reinterpret_cast<float2*>(ored + (w8 * kHeads + 0) * kRank + lane * 8)[c] = acc0[c];
        reinterpret_cast<float2*>(ored + (w8 * kHeads + 1) * kRank + lane * 8)[c] = acc1[c];
      }
      tc::named_bar(7, 2 * kWg);
      const int t2 = threadIdx.x - 3 * kWg;   // 0..255
#pragma unroll
      for (int j = 0; j < kHeads; ++j) {
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) o += ored[(k * kHeads + j) * kRank + t2];
        const int64_t bh = (int64_t)b * a.n_heads + head0 + j;
        a.part_o[(bh * a.n_splits + split) * kRank + t2] = o;
      }
      if (Y == 0 && ei < kHeads) {
        float L = 0.f;
        for (int k = 0; k < 4; ++k) L += (ei == 0) ? lred[k].x : lred[k].y;
        const int64_t bh = (int64_t)b * a.n_heads + head0 + ei;
        a.part_ml[bh * a.n_splits + split] = make_float2(ei == 0 ? m_run0 : m_run1, L);
      }
    }
  } else {
    // ------------------------------------------------------------ int4 key converter (I4K only)
    // thread = one token row: expand the row's packed codes into exact fp16 codes in the MMA
    // operand ring (128-byte swizzle, one 64-column chunk per stage).
    if constexpr (I4K) {
      setmaxnreg_dec<LY::kRegsConv>();
      const int r = threadIdx.x - 5 * kWg;
      bool ok = true;
      for (int it = 0; it < n_tiles && ok; ++it) {
        const int ps = it % kPStages;
        if (!tc::mbar_wait_bounded(&pfull[ps], (it / kPStages) & 1, abort_flag, kWaitNs)) break;
        const uint8_t* prow = smem + LY::kOffPk + ps * LY::kPStage + r * 128;
        for (int kc = 0; kc < kChunks; ++kc) {
          const int si = it * kChunks + kc;
          const int stage = si % kStages;
          if (!tc::mbar_wait_bounded(&emptyA[stage], ((si / kStages) & 1) ^ 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          convert_int4_row_chunk(prow, smem + LY::kOffA + stage * kAStage + r * 128, r, kc);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&fullA[stage]);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&pempty[ps]);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_error(a.err, kCodeTimeout, kErrWait, blockIdx.x, b);
  if (warp == 1) tc::tmem_dealloc(tmem_base, kTmemCols);
  merge_if_last(a, b, head0, kHeads, reinterpret_cast<volatile int*>(smem + LY::kOffMisc + 8),
                reinterpret_cast<float*>(smem + LY::kOffV));  // the H_v ring is free by now
}

// ---------------------------------------------------------------------------- host side

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

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, dt, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tma_available() { return encode_fn() != nullptr; }

bool tma_encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  return encode_fn() != nullptr && encode(m, dt, rank, base, dims, strides, box, sw);
}

bool tc_supported(const DecodeArgs& a) {
  const bool i4 = a.k_dtype == kINT4;
  // key and value latents of one dtype, or fp16 / bf16 keys with int4 values (V-only int4)
  const bool types = (a.k_dtype == kF16 || a.k_dtype == kBF16 || i4) &&
                     (a.v_dtype == a.k_dtype || (!i4 && a.v_dtype == kINT4));
  return types && (!i4 || a.bk_dtype == kF16) && a.dh == kDh && a.rk == kRank && a.rv == kRank &&
         a.s % kHeads == 0 &&
         (int64_t)a.batch * a.capacity >= kTile && (int64_t)a.batch * a.capacity < (int64_t(1) << 31) &&
         encode_fn() != nullptr;
}

int tc_tile_tokens() { return kTile; }
int tc_ctas_per_group(const DecodeArgs& a) { return a.s / kHeads; }

template <typename VT, bool I4K, bool FOLD>
cudaError_t launch_variant(const CUtensorMap& tm_hk, const CUtensorMap& tm_hv, const CUtensorMap& tm_b,
                           const TcParams& P, cudaStream_t st) {
  using LY = Lay<I4K, std::is_same<VT, Int4>::value>;
  auto kern = decode_tc_kernel<VT, I4K, FOLD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmemAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid(P.a.n_splits * P.hp_count, P.a.n_g, P.a.batch);
  kern<<<grid, LY::kThreads, LY::kSmemAlloc, st>>>(tm_hk, tm_hv, tm_b, P);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  const bool i4k = a.k_dtype == kINT4, i4v = a.v_dtype == kINT4;
  const CUtensorMapDataType dt = a.k_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tm_hk, tm_hv, tm_b;
  const cuuint64_t rows = (cuuint64_t)a.batch * a.capacity;
  // packed int4 rows [rows][n_g][r/2] bytes; fp16 / bf16 rows [rows][n_g][r]
  const cuuint64_t pdims[3] = {(cuuint64_t)kRank / 2, (cuuint64_t)a.n_g, rows};
  const cuuint64_t pstrides[2] = {(cuuint64_t)kRank / 2, (cuuint64_t)a.n_g * (kRank / 2)};
  const cuuint64_t fdims[3] = {(cuuint64_t)kRank, (cuuint64_t)a.n_g, rows};
  const cuuint64_t fstrides[2] = {(cuuint64_t)kRank * 2, (cuuint64_t)a.n_g * kRank * 2};
  if (i4k) {
    // H_k as whole 128-token packed tiles, 128-byte swizzle for the converter's row reads
    const cuuint32_t boxk[3] = {kRank / 2, 1, kTile};
    if (!encode(&tm_hk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.hk, pdims, pstrides, boxk, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    // H_k as boxes of 64 ranks x 1 group x 128 tokens, 128-byte swizzle (the MMA operand)
    const cuuint32_t boxk[3] = {kKChunk, 1, kTile};
    if (!encode(&tm_hk, dt, 3, a.hk, fdims, fstrides, boxk, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  if (i4v) {
    // H_v as 64-token chunks of packed rows, unswizzled (row reads)
    const cuuint32_t boxv[3] = {kRank / 2, 1, 64};
    if (!encode(&tm_hv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.hv, pdims, pstrides, boxv, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    // H_v as whole 512-byte rows x 32 tokens, unswizzled (row reads)
    const cuuint32_t boxv[3] = {(cuuint32_t)kRank, 1, (cuuint32_t)Lay<false, false>::kVTok};
    if (!encode(&tm_hv, dt, 3, a.hv, fdims, fstrides, boxv, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
  }
  {
    // B_k^T as [n_g * s * d_h][r]: boxes of 64 ranks x 256 rows, 128-byte swizzle
    const cuuint64_t dims[2] = {(cuuint64_t)a.rk, (cuuint64_t)a.n_g * a.s * a.dh};
    const cuuint64_t strides[1] = {(cuuint64_t)a.rk * 2};
    const cuuint32_t box[2] = {kKChunk, kN};
    if (!encode(&tm_b, i4k ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : dt, 2, a.bkt, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  TcParams P;
  P.a = a;
  P.hp_count = a.s / kHeads;
  P.bf16 = a.k_dtype == kBF16;
  // fp16 operands carry the folded query with 11-bit precision; bf16 ones (8-bit) would not,
  // so the bf16 kernel rebuilds K exactly and applies the query in the epilogue
  if (i4k) return launch_variant<Int4, true, true>(tm_hk, tm_hv, tm_b, P, st);
  if (a.k_dtype == kBF16)
    return i4v ? launch_variant<Int4, false, false>(tm_hk, tm_hv, tm_b, P, st)
               : launch_variant<__nv_bfloat16, false, false>(tm_hk, tm_hv, tm_b, P, st);
  return i4v ? launch_variant<Int4, false, true>(tm_hk, tm_hv, tm_b, P, st)
             : launch_variant<__half, false, true>(tm_hk, tm_hv, tm_b, P, st);
}

// ---------------------------------------------------------------------------- int4 test exports
// Both kernels below run the int4 routines of decode_tc_kernel<Int4> itself (the same device
// functions), so that their outputs can be compared bit for bit with the oracle.

namespace {

constexpr int kDbgPk = 0;                        // packed tile (128 tokens x 128 B), 1024-aligned
constexpr int kDbgOp = kTile * (kRank / 2);      // fp16 operand: kChunks x 16 KB
constexpr int kDbgBar = kDbgOp + kChunks * kAStage;
constexpr int kDbgSmem = kDbgBar + 16 + 1024;

// Key side: TMA loads a packed 128-token tile with the 128-byte swizzle, exactly as the decode
// kernel's producer does; thread r converts row r with the converter routine into the swizzled
// fp16 operand layout and reads its own row back, writing the operand values in the operand's
// rank order and, in fp32, operand value x key scale.
__global__ void __launch_bounds__(kTile) debug_int4_operand_kernel(const __grid_constant__ CUtensorMap tm_hk,
                                                                   const __half* k_scale, int64_t capacity, int n_g,
                                                                   int64_t n_tokens, uint16_t* codes, float* deq,
                                                                   ErrWord* err, uint64_t wait_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kDbgBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kDbgBar + 8);
  const int r = threadIdx.x;
  const int t0 = blockIdx.x * kTile, g = blockIdx.y, b = blockIdx.z;
  if (r == 0) {
    tc::mbar_init(bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (r == 0) {
    tc::mbar_arrive_expect_tx(bar, kTile * (kRank / 2));
    tc::tma_load_3d(smem + kDbgPk, &tm_hk, bar, 0, g, int(b * capacity + t0));
  }
  if (!tc::mbar_wait_bounded(bar, 0, abort_flag, wait_ns)) {
    volatile int quiet = 0;
    tc::mbar_wait_bounded(bar, 0, &quiet, wait_ns);   // the copy may still land: let it
    if (r == 0) record_error(err, kCodeTimeout, kErrWait, blockIdx.x, b);
    return;
  }
  uint8_t* arow_base = smem + kDbgOp + r * 128;
  for (int kc = 0; kc < kChunks; ++kc) convert_int4_row_chunk(smem + kDbgPk + r * 128, arow_base + kc * kAStage, r, kc);
  const int64_t t = t0 + r;
  if (t >= n_tokens) return;
  const float s = __half2float(k_scale[((int64_t)b * capacity + t) * n_g + g]);
  const int64_t o = (((int64_t)b * n_tokens + t) * n_g + g) * kRank;
  for (int kc = 0; kc < kChunks; ++kc) {
    for (int j = 0; j < 8; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(arow_base + kc * kAStage + ((j ^ (r & 7)) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const int64_t c0 = o + kc * kKChunk + j * 8;
      for (int e = 0; e < 8; ++e) {
        const uint16_t bits = uint16_t(w[e >> 1] >> (16 * (e & 1)));
        codes[c0 + e] = bits;
        if (deq) deq[c0 + e] = __half2float(__ushort_as_half(bits)) * s;
      }
    }
  }
}

// Value side: one warp per (16-token block, group, batch row) runs the dp2a routine of the decode
// kernel's p H_v over the block with the caller's 15-bit integer weights, and writes the exact
// int32 sums sum_t w[t][head] code[t][c] for both heads.
__global__ void debug_int4_dp2a_kernel(const uint8_t* cache, int64_t capacity, int n_g, int64_t n_tokens,
                                       const int32_t* weights, int32_t* sums) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int g = blockIdx.y, b = blockIdx.z;
  const int64_t nblk = (n_tokens + 15) / 16;
  if (blk >= nblk) return;   // warp-uniform
  const int jt = lane & 15, hh = lane >> 4;
  const int64_t tq = blk * 16 + jt;
  const uint32_t qv = tq < n_tokens ? uint32_t(weights[((int64_t)b * n_tokens + tq) * 2 + hh]) : 0u;
  uint32_t qpair, qsum;
  dp2a_pack_weights(qv, qpair, qsum);
  uint32_t ai[2][8];
#pragma unroll
  for (int c = 0; c < 8; ++c) ai[0][c] = ai[1][c] = 0u;
  for (int ch = 0; ch < 2; ++ch) {
    uint32_t u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t t = blk * 16 + ch * 8 + k;
      u[k] = t < n_tokens
                 ? *reinterpret_cast<const uint32_t*>(cache + (((int64_t)b * capacity + t) * n_g + g) * (kRank / 2) +
                                                      lane * 4)
                 : 0u;
    }
    dp2a_accumulate8(u, qpair, ch, ai);
  }
  const uint32_t qs0 = __shfl_sync(0xffffffffu, qsum, 0), qs1 = __shfl_sync(0xffffffffu, qsum, 16);
  int32_t* o = sums + ((((int64_t)b * nblk + blk) * n_g + g) * 2) * kRank + lane * 8;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    o[c] = dp2a_unbias(ai[0][c], qs0);
    o[kRank + c] = dp2a_unbias(ai[1][c], qs1);
  }
}

}  // namespace

bool tc_int4_debug_supported(int n_g, int rank, int64_t rows) {
  return rank == kRank && n_g > 0 && rows >= kTile && rows < (int64_t(1) << 31) && encode_fn() != nullptr;
}

cudaError_t launch_debug_int4_operand(const void* hk, const __half* k_scale, int64_t capacity, int n_g, int batch,
                                      int64_t n_tokens, uint16_t* codes, float* deq, ErrWord* err,
                                      cudaStream_t st) {
  if (!tc_int4_debug_supported(n_g, kRank, (int64_t)batch * capacity)) return cudaErrorNotSupported;
  if (n_tokens == 0 || batch == 0) return cudaSuccess;
  CUtensorMap tm;
  const cuuint64_t dims[3] = {(cuuint64_t)kRank / 2, (cuuint64_t)n_g, (cuuint64_t)batch * capacity};
  const cuuint64_t strides[2] = {(cuuint64_t)kRank / 2, (cuuint64_t)n_g * (kRank / 2)};
  const cuuint32_t box[3] = {kRank / 2, 1, kTile};   // the decode kernel's H_k box and swizzle
  if (!encode(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, hk, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(debug_int4_operand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDbgSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((n_tokens + kTile - 1) / kTile), (unsigned)n_g, (unsigned)batch);
  debug_int4_operand_kernel<<<grid, kTile, kDbgSmem, st>>>(tm, k_scale, capacity, n_g, n_tokens, codes, deq, err,
                                                          1000000000ull);
  return cudaGetLastError();
}

cudaError_t launch_debug_int4_dp2a(const void* cache, int64_t capacity, int n_g, int batch, int64_t n_tokens,
                                   const int32_t* weights, int32_t* sums, cudaStream_t st) {
  if (n_tokens == 0 || batch == 0) return cudaSuccess;
  const int64_t nblk = (n_tokens + 15) / 16;
  const int warps = 4;
  dim3 grid((unsigned)((nblk + warps - 1) / warps), (unsigned)n_g, (unsigned)batch);
  debug_int4_dp2a_kernel<<<grid, warps * 32, 0, st>>>(static_cast<const uint8_t*>(cache), capacity, n_g, n_tokens,
                                                      weights, sums);
  return cudaGetLastError();
}

}  // namespace palu
