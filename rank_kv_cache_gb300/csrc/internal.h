// Internal interface between the C ABI (palu_host.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace palu {

// Everything a decode launch needs, flattened to plain pointers and sizes.
struct DecodeArgs {
  // latent cache
  const void* hk;
  const void* hv;
  const __half* k_scale;
  const __half* v_scale;
  int64_t capacity;
  // shapes and types
  int n_heads, n_g, s, dh, rk, rv;
  int k_dtype, v_dtype, bk_dtype;
  // per call
  const int32_t* seq_lens;
  const int32_t* positions;   // nullable
  int batch;
  int max_seq_len;
  int64_t max_pos;
  // workspace-resident operands
  const float* qbuf;          // [B][n][dh] rotated (rope) or [B][n][rk] absorbed; pre-scaled by log2(e)/sqrt(dh)
  const void* bk;             // [n_g][rk][s*dh], bk_dtype
  const void* bkt;            // [n_g][s*dh][rk], MMA dtype: the K-major tcgen05 operand, rows of each head
                              // pair interleaved by head, ranks permuted in eights for int4 caches
  const float2* rope;         // [max_pos][dh/2] (cos, sin)
  const uint64_t* phase;      // [dh/2] frequency of each pair as a 64-bit fraction of a turn
  // query (read directly by kernels that rotate it themselves)
  const void* q;
  int q_dtype;
  const int32_t* q_pos;       // nullable
  float qscale;               // log2(e) / sqrt(dh)
  // split-T partials
  float* part_o;              // [B][n][n_splits][rv]
  float2* part_ml;            // [B][n][n_splits] (running max m in log2 units, sum l)
  int n_splits;
  int tiles_per_split;
  ErrWord* err;
  // In-kernel split merge: when `counters` is set, the last CTA of each unit (counted with
  // an atomic that it resets afterwards) merges that unit's partials into out / lse, and no
  // merge kernel is launched. counters: [max_batch][n_heads], zero between calls.
  unsigned* counters;
  float* out;                 // [B][n][out_rv ? out_rv : rv]
  float* lse;
  // Packed groups (out_rv > 0): the kernels run groups of four heads whose rv = 256 latent
  // columns hold 4 / pack_s source groups of out_rv ranks each; head h's output is the slice of
  // its own source group, columns ((h % 4) / pack_s) * out_rv + [0, out_rv).
  int out_rv;
  int pack_s;
  // Split groups (g_split > 1, absorbed path): each cache group of g_split * 4 heads is run as g_split
  // kernel groups of four heads over the same latents; kernel group g reads cache group g / g_split
  // of the n_g / g_split in the cache.
  int g_split;
  // failure-detection test hook (PALU_FLAG_TEST_STALL): the tensor-core kernel's H_v
  // producer issues nothing; wait_ns bounds every mbarrier wait of that kernel
  int test_stall;
  uint64_t wait_ns;
  // ALiBi (absorbed path): every score of head i gets m_i (pos_t - q_pos), m_i = 2^(-8 (i + 1) / n)
  int alibi;
};

// create-time set-up
cudaError_t launch_rope_table(float2* tab, uint64_t* phase, int64_t max_pos, int dh, double theta, cudaStream_t st);
cudaError_t launch_copy_bk(const void* src, int bk_dtype, void* dst, void* dst_t, int mma_dtype, int n_g,
                           int rk, int cols, int dh, int perm8, int pack, int split, int src_s, int src_rk,
                           cudaStream_t st);

// per-call kernels
cudaError_t launch_qprep(int mode, const void* q, int q_dtype, const DecodeArgs& a, const int32_t* q_pos,
                         float qscale, float* qbuf, cudaStream_t st);
cudaError_t launch_decode_simt(int mode, const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_combine(const DecodeArgs& a, float* out, float* lse, cudaStream_t st);
// append the new tokens' key and value latents in one launch
cudaError_t launch_append(void* cache_k, __half* scale_k, int rank_k, const void* src_k, void* cache_v,
                          __half* scale_v, int rank_v, const void* src_v, int k_dtype, int v_dtype, int64_t capacity,
                          int n_g, int src_dtype, const int32_t* dst_slot, int batch, int n_new, ErrWord* err,
                          cudaStream_t st);
cudaError_t launch_debug_dequant(const void* cache, const __half* scale, int cache_dtype, int64_t capacity,
                                 int n_g, int rank, int batch, int64_t n_tokens, float* out, cudaStream_t st);

// tcgen05 rebuild path (decode_tc.cu); returns cudaErrorNotSupported when the shape has no kernel
bool tc_supported(const DecodeArgs& a);
int tc_tile_tokens();
int tc_ctas_per_group(const DecodeArgs& a);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
// int4 test exports that run the tensor-core kernel's own converter and dp2a routines
bool tc_int4_debug_supported(int n_g, int rank, int64_t rows);
cudaError_t launch_debug_int4_operand(const void* hk, const __half* k_scale, int64_t capacity, int n_g, int batch,
                                      int64_t n_tokens, uint16_t* codes, float* deq, ErrWord* err, cudaStream_t st);
cudaError_t launch_debug_int4_dp2a(const void* cache, int64_t capacity, int n_g, int batch, int64_t n_tokens,
                                   const int32_t* weights, int32_t* sums, cudaStream_t st);

// cuTensorMapEncodeTiled through the runtime's driver entry point (decode_tc.cu); false when the
// driver offers no entry point or rejects the map
bool tma_available();
bool tma_encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw);

// latent production H = x A on tcgen05 (prefill.cu)
struct ProjectArgs {
  void* cache[2];             // key and value latent caches
  __half* scale[2];           // int4 scales (nullable otherwise)
  int cache_dtype;
  int64_t capacity;
  int n_g, rank;
  int64_t d;                  // d_model
  const int32_t* dst_slot;    // [batch]
  int n_new;
  int64_t M;                  // batch * n_new rows of x
  ErrWord* err;
  uint64_t wait_ns;
};
cudaError_t launch_project_latents(const void* x, const void* w, int bf16, const ProjectArgs& a, cudaStream_t st);
cudaError_t launch_prepare_down_proj(const void* a_k, const void* a_v, int a_dtype, int n_g, int rank, int64_t d,
                                     int w_dtype, void* w, cudaStream_t st);

// hybrid cache: the dense segment merged with the latent middle's decode (hybrid.cu)
struct DenseArgs {
  const void* k;              // [rows][capacity][n_heads][dh] dense keys (rotated at their positions on the RoPE path)
  const void* v;              // same layout, values
  int dtype;                  // kF32, kF16 or kBF16
  const int32_t* n_tokens;    // [batch] dense tokens per row
  int64_t capacity;
  int n_heads, dh, rv, batch;
  int rope;                   // rotate the query at q_pos
  const int32_t* q_pos;
  const float2* rope_tab;     // [max_pos][dh/2]
  int64_t max_pos;
  const void* q;
  int q_dtype;
  float qscale;               // log2(e) / sqrt(dh)
  float* out;                 // [batch][n_heads][rv]: the middle's output, rescaled in place
  float* out_dense;           // [batch][n_heads][dh]
  float* lse;                 // [batch][n_heads]: the middle's lse in, the merged lse out
  ErrWord* err;
};
cudaError_t launch_merge_dense(const DenseArgs& d, cudaStream_t st);

// page-factorised decode (paged.cu): PuzzleKV pages of P = 32 tokens, d_h = 128, rank 8, 16 or 32
struct PagedArgs {
  const void* pages;          // [rows][capacity][n_heads] records: L_K [P][r], R_K [r][d], L_V [P][r], R_V [r][d]
  const int32_t* n_pages;     // [batch] factorised pages per row
  int64_t capacity;           // pages per row
  int max_pages;              // bound on n_pages (this call)
  int dtype;                  // kF16 or kBF16
  int rank;
  int n_heads;
  int rope;                   // rotate the query at q_pos
  const int32_t* q_pos;
  const float2* rope_tab;     // [max_pos][d/2]
  int64_t max_pos;
  const void* q;
  int q_dtype;
  float qscale;               // log2(e) / sqrt(d)
  int pages_per_split;
  ErrWord* err;
  uint64_t wait_ns;
  DecodeArgs m;               // the split merge: batch, n_heads, n_splits, rv = d, part_o, part_ml, counters, out, lse
};
int paged_ctas_per_sm(int rank);
cudaError_t launch_decode_paged(const PagedArgs& P, cudaStream_t st);

// TMA-streaming absorbed-mode kernel (decode_abs.cu)
bool abs_supported(const DecodeArgs& a);
int abs_stage_tokens();
cudaError_t launch_decode_abs(const DecodeArgs& a, cudaStream_t st);

constexpr int kSimtTile = 16;   // tokens per SIMT tile

}  // namespace palu
