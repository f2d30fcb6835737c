/*
 * palu_attn.h -- C ABI for Palu-style group-head low-rank (G-LRD) decode
 * attention over a latent KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The operation ("Palu: KV-Cache Compression With Low-Rank Projection", method
 * section "方法细节"):
 *   - The key/value projections of each group of s consecutive heads are
 *     factored offline, W_g ~= A_g B_g (truncated SVD, "背景知识"), and only the
 *     latents h_g = x A_g (r values per token and group) are cached.
 *   - RoPE models: each head's keys are rebuilt on chip from the cached latents,
 *     K = H_k,g B_k,g[:, head block], rotated by RoPE at every token's own
 *     position, and scored against the rotated query (RoPE paragraph and the
 *     online-rebuild kernel paragraph of "补充细节").
 *   - Non-RoPE models: the query is absorbed, q' = q B_k^T, and scored straight
 *     against H_k (key-fusion paragraph).
 *   - Softmax over all cached tokens, then p is applied to the value latents,
 *     o = p H_v, so the output stays in latent space: B_v is fused into W_o
 *     offline (value-fusion paragraph).
 *   - Optionally the latents are stored as per-token int4 codes with an fp16
 *     scale; a Walsh-Hadamard rotation folded into A and B beforehand needs no
 *     run-time work (Hadamard paragraph).
 *
 * Conventions fixed by this library (the pages leave them open):
 *   - Row vectors: h = x A, A in R^{d x r}. Head i is column block (i % s) of
 *     group (i / s).
 *   - Score scale 1/sqrt(d_h) on both paths.
 *   - RoPE is rotate-half: pairs (k, k + d_h/2) rotated by pos * theta^(-2k/d_h).
 *   - The query is passed UNROTATED; it is rotated at q_pos, which defaults to
 *     the position of the last cached token. No causal mask.
 *   - int4 codes: symmetric in [-7, 7], one fp16 scale per token and group,
 *     scale = fp16_rn(min(amax / 7, 65504)) with IEEE fp32 division,
 *     code = rint_half_even(h / scale) clamped to [-7, 7]; element 2j in the low
 *     nibble and 2j+1 in the high nibble of byte j (two's complement).
 *
 * Memory: every pointer argument that the comments call "device" is device
 * memory owned by the caller, and must stay valid until the work queued on the
 * given stream has finished. The library allocates no device memory: scratch
 * lives in the caller-provided workspace. A handle owns host memory only.
 *
 * Concurrency: the decode calls of one handle (palu_decode_attn, _hybrid, _paged)
 * share its workspace (split partials, the split-merge counters, the error word);
 * calls that may overlap on the GPU need one handle, with its own workspace, each.
 * Calls queued on one stream are ordered and safe.
 *
 * Errors: every call returns a palu_status_t; nothing aborts, prints or throws.
 * Argument checks happen on the host before anything is queued. Conditions only
 * the GPU can see (a position outside the RoPE table, a sequence longer than
 * the cache, a bounded wait that gave up) are recorded in an error word inside
 * the workspace; the kernels clamp the offending index and carry on, and
 * palu_attn_check reports (and clears) it. No other call synchronises.
 *
 * Threading: calls on one handle must not overlap (they share one workspace).
 * Different handles are independent.
 */
#ifndef PALU_ATTN_H
#define PALU_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PALU_ABI_VERSION 1

/* A CUDA stream. Pass a cudaStream_t (or CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* palu_stream_t;

typedef enum palu_status_t {
  PALU_OK = 0,
  PALU_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size, inconsistent descriptor */
  PALU_ERR_UNSUPPORTED = 2,  /* a valid shape or dtype combination this build has no kernel for
                                (shapes the descriptor accepts but no fast kernel covers are not
                                refused: they run on the CUDA-core kernel, see palu_decode_plan) */
  PALU_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  PALU_ERR_DEVICE = 4,       /* a kernel recorded an out-of-range index in the error word */
  PALU_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (error word) */
  PALU_ERR_WORKSPACE = 6     /* workspace missing, too small or not 256-byte aligned */
} palu_status_t;

typedef enum palu_dtype_t {
  PALU_F32 = 0,
  PALU_F16 = 1,
  PALU_BF16 = 2,
  PALU_INT4 = 3   /* latents only: packed codes + fp16 per-token scales */
} palu_dtype_t;

typedef enum palu_mode_t {
  PALU_MODE_ROPE = 0,      /* rebuild K = H_k B_k on chip, rotate, score */
  PALU_MODE_ABSORBED = 1   /* score q B_k^T straight against H_k (no RoPE) */
} palu_mode_t;

typedef struct palu_attn_desc {
  int abi_version;        /* must be PALU_ABI_VERSION */
  int n_heads;            /* n */
  int head_dim;           /* d_h: 64 or 128 */
  int group_size;         /* s: 1, 2, 4 or 8 (M-LRD is s = 1); 16 or 32 (up to J-LRD, s = n) on the
                             RoPE path with head_dim 128, ranks 256 and F16/BF16/INT4 latents
                             ("方法细节", M-LRD / G-LRD / J-LRD paragraphs); n_heads % s == 0.
                             s = 1 or 2 with ranks 64 s, head_dim 128, F16/BF16 latents and
                             n_heads % 4 == 0 run packed four heads at a time with a block-diagonal
                             B_k (the workspace then holds 4 / s times the B_k bytes); the output
                             layout is unchanged ([batch][n_heads][rank_v]). On the absorbed path
                             s = 8, 16 or 32 at ranks 256 with F16/BF16 latents run as s / 4 groups
                             of four heads over the same cached latents */
  int rank_k;             /* r_k per group: 64, 128 or 256 */
  int rank_v;             /* r_v per group: 64, 128 or 256 */
  palu_dtype_t k_dtype;   /* key-latent storage */
  palu_dtype_t v_dtype;   /* value-latent storage: k_dtype, or PALU_INT4 under F16 / BF16 keys
                             (int4 values only, the Palu notes' 4-bit V setting, "实验结果") */
  palu_dtype_t bk_dtype;  /* B_k storage: equals k_dtype, or PALU_F16 when k_dtype is PALU_INT4 */
  palu_dtype_t q_dtype;   /* query storage: F32, F16 or BF16 */
  palu_mode_t mode;
  double rope_theta;      /* RoPE base (e.g. 10000); ignored by the absorbed mode */
  int max_batch;          /* largest batch any decode call will pass */
  int64_t max_tokens;     /* largest sequence length any decode call will see */
  int64_t max_position;   /* positions must lie in [0, max_position); 0 means max_tokens */
  uint32_t flags;         /* 0, PALU_FLAG_ALIBI, or PALU_FLAG_TEST_STALL (test builds of callers only) */
} palu_attn_desc;

/*
 * Failure-detection test hook; the pages have no counterpart. With this flag the
 * tensor-core RoPE kernel's H_v producer issues no loads, so the consumers' bounded
 * waits give up (after 50 ms instead of the normal 1 s), every CTA drains its copies,
 * frees its tensor memory and returns, and the next palu_attn_check reports
 * PALU_ERR_TIMEOUT. Outputs of such a call are undefined. The other kernels ignore it
 * (palu_decode_plan tells which kernel a call uses). Never set it in production.
 */
#define PALU_FLAG_TEST_STALL 0x80000000u

/*
 * ALiBi position bias on the absorbed path ("方法细节", key-fusion paragraph: a position
 * encoding that never touches the keys, ALiBi being the example, leaves the absorbed query
 * valid). Each score of head i gets -m_i (q_pos - pos_t) with the slopes m_i = 2^(-8 (i + 1) / n)
 * of the ALiBi paper the notes cite; pos_t comes from `positions` (default t) and q_pos from
 * `q_pos` (default the last cached token's position). Only with PALU_MODE_ABSORBED (else
 * PALU_ERR_INVALID_ARG); palu_decode_attn_noalloc and palu_decode_hybrid take no positions and
 * return PALU_ERR_UNSUPPORTED for it.
 */
#define PALU_FLAG_ALIBI 0x1u

/*
 * A latent cache, caller-owned device memory. With n_g = n_heads / group_size:
 *   hk       [max_rows][capacity][n_g][rank_k] elements of k_dtype
 *            (PALU_INT4: [max_rows][capacity][n_g][rank_k / 2] bytes)
 *   hv       [max_rows][capacity][n_g][rank_v] elements of v_dtype (same rule)
 *   k_scale  PALU_INT4 only: [max_rows][capacity][n_g] fp16 scales, else NULL
 *   v_scale  PALU_INT4 only: same for hv, else NULL
 * Batch element b of a call uses row b. hk and hv must be 16-byte aligned.
 */
typedef struct palu_cache {
  void* hk;
  void* hv;
  void* k_scale;
  void* v_scale;
  int64_t capacity;       /* tokens per row (the token stride) */
} palu_cache;

typedef struct palu_attn* palu_attn_t;

/* Bytes of device workspace palu_attn_create needs for this descriptor. */
palu_status_t palu_attn_workspace_size(const palu_attn_desc* desc, size_t* bytes);

/*
 * Create a handle. B_k is device memory [n_g][rank_k][group_size * head_dim]
 * row-major in desc->bk_dtype: the per-group reconstruction factor B_g of the
 * G-LRD factorisation ("方法细节", G-LRD paragraph), already Hadamard-folded if
 * the latents were rotated. It is copied (and re-laid out) into the workspace
 * on `stream`, together with a RoPE cos/sin table computed in float64, so B_k
 * may be freed once that stream has passed this call. `workspace` (device,
 * 256-byte aligned, at least palu_attn_workspace_size bytes) must outlive the
 * handle. The handle itself is host memory.
 */
palu_status_t palu_attn_create(const palu_attn_desc* desc, const void* B_k, void* workspace,
                               size_t workspace_bytes, palu_stream_t stream, palu_attn_t* out);

/*
 * Append n_new tokens per batch row to the cache ("方法细节": the latents h = x A
 * are what is stored). hk_new [batch][n_new][n_g][rank_k] and hv_new
 * [batch][n_new][n_g][rank_v] are device arrays of src_dtype (F32, F16 or BF16).
 * dst_slot (device, [batch] int32) gives the first token index written in each
 * row; tokens dst_slot[b] .. dst_slot[b] + n_new - 1 are overwritten. Float
 * caches store the values rounded to nearest; int4 caches quantise them per
 * token and group (convention in the file header). An index past the capacity
 * is recorded in the error word and the row is skipped.
 */
palu_status_t palu_append_latents(palu_attn_t h, const palu_cache* cache, const void* hk_new,
                                  const void* hv_new, palu_dtype_t src_dtype, const int32_t* dst_slot,
                                  int batch, int n_new, palu_stream_t stream);

/*
 * Decode attention for one new query per batch row.
 *   q          device [batch][n_heads][head_dim], desc->q_dtype, unrotated
 *   seq_lens   device [batch] int32: tokens 0 .. seq_lens[b]-1 of row b attend
 *   positions  device [batch][capacity] int32 RoPE positions, or NULL for
 *              position = token index (ignored by the absorbed mode)
 *   q_pos      device [batch] int32 query positions, or NULL for the position of
 *              the last cached token (ignored by the absorbed mode)
 *   max_seq_len host upper bound on every seq_lens[b] (<= desc->max_tokens and
 *              <= cache->capacity); it sizes the launch. A larger seq_lens[b] is
 *              clamped and recorded in the error word.
 *   out        device [batch][n_heads][rank_v] float32: o_i = p_i H_v,g
 *   lse        device [batch][n_heads] float32 natural log-sum-exp of the scaled
 *              scores, or NULL. An empty row (seq_lens[b] == 0) yields o = 0 and
 *              lse = -inf.
 * Asynchronous on `stream`. Kernel choice: RoPE mode with fp16/bf16/int4 latents,
 * head_dim 128, rank 256 and an even group size runs the tensor-core rebuild kernel;
 * absorbed mode with fp16/bf16 latents, group size 4 and rank 256 runs the TMA
 * streaming kernel; every other accepted descriptor (fp32 latents, int4 absorbed,
 * group size 1, head_dim 64, ranks 64/128) runs the CUDA-core kernel, which is
 * correct for all of them but not tuned. palu_decode_plan reports the choice.
 */
palu_status_t palu_decode_attn(palu_attn_t h, const void* q, const palu_cache* cache,
                               const int32_t* seq_lens, const int32_t* positions, const int32_t* q_pos,
                               int batch, int64_t max_seq_len, float* out, float* lse,
                               palu_stream_t stream);

/*
 * Which kernel palu_decode_attn would launch for this shape, and its split-T plan.
 * Host-only: reads no device memory and queues nothing. A convenience for tests and
 * benchmarks; the pages' statement of the problem has no such call.
 *   cache_capacity  tokens per batch row of the cache that would be passed
 *   batch, max_seq_len  as for palu_decode_attn (same limits)
 *   kernel    out: a palu_kernel_t
 *   n_splits  out: split-T ranges per (batch row, head group); 1 = no split
 *   launches  out: kernel launches the decode call makes (the query preparation
 *             of the CUDA-core and absorbed kernels counts as one)
 * PALU_ERR_INVALID_ARG on a NULL pointer or an argument outside the limits.
 */
typedef enum {
  PALU_KERNEL_TC_ROPE = 1,       /* tensor-core rebuild + RoPE (fp16, bf16, int4 latents) */
  PALU_KERNEL_TMA_ABSORBED = 2,  /* absorbed query, TMA-streamed latents (fp16, bf16) */
  PALU_KERNEL_SIMT = 3           /* CUDA-core kernel: every other supported combination */
} palu_kernel_t;
palu_status_t palu_decode_plan(palu_attn_t h, int64_t cache_capacity, int batch, int64_t max_seq_len,
                               int* kernel, int* n_splits, int* launches);

/*
 * Absorbed-mode decode for callers that cannot allocate device memory (a plugin
 * whose host owns every allocation, an engine with a fixed memory plan, code that
 * must not allocate once serving starts). The pages have no counterpart to it.
 * It takes no handle and no workspace: B_k (device, [n_g][rank_k][s * head_dim]
 * in desc->bk_dtype) and the query are read directly, and the scratch (error
 * word, absorbed queries, split partials) lives in one fixed 8 MiB device array
 * inside this library, which every GPU that loads the library holds until the
 * process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - desc->mode must be PALU_MODE_ABSORBED (else PALU_ERR_UNSUPPORTED);
 *     arguments as for palu_decode_attn, without positions and q_pos.
 *   - A request whose scratch (4 bytes x batch x n_heads x (rank_k + rank_v) for
 *     one split, plus alignment) does not fit in 8 MiB returns PALU_ERR_WORKSPACE
 *     before anything is queued; larger T only lowers the split count.
 *   - The device is the calling thread's current device, and `stream` must belong
 *     to it (else PALU_ERR_INVALID_ARG). The first call on a device looks up the
 *     array's address on that device (cudaGetSymbolAddress), so make that first
 *     call before any stream capture.
 *   - int4 latents need k_scale / v_scale as for palu_decode_attn (non-NULL, 2-byte
 *     aligned, for each int4 side).
 *   - Every call shares the one array, and its contents persist between calls;
 *     the error word is cleared at the start of each call. Calls that overlap on
 *     the GPU (different streams, or host threads racing) race on the scratch:
 *     serialise them. Out-of-range sequence lengths are clamped; there is no
 *     handle through which to report them.
 */
palu_status_t palu_decode_attn_noalloc(const palu_attn_desc* desc, const void* B_k, const void* q,
                                       const palu_cache* cache, const int32_t* seq_lens, int batch,
                                       int64_t max_seq_len, float* out, float* lse, palu_stream_t stream);

/*
 * The layer's output projection from the latent decode outputs, with B_v fused into
 * W_o ("方法细节", value-fusion paragraph: head i's output p_i V_i = p_i H_v,g B_v^(i)
 * only meets its own rows W_o^(i), so V is never rebuilt):
 *   y[b] = sum_i o[b][i] W_f^(i),   W_f^(i) = B_v^(i) W_o^(i)   (rank_v x d_model).
 *
 * palu_fuse_value_output forms the fused weight once (an offline transform), on the
 * current device:
 *   B_v      device [n_g][rank_v][group_size * head_dim] in in_dtype (F32, F16, BF16),
 *            the per-group value factor; head i uses column block i % s of group i / s
 *   W_o      device [n_heads * head_dim][d_model] in in_dtype, row-major (the rows of
 *            head i are i * head_dim .. (i + 1) * head_dim - 1)
 *   W_fused  device [n_heads * rank_v][d_model] in out_dtype (F16 or BF16): head i's
 *            block is rows i * rank_v .. (i + 1) * rank_v - 1; fp32 accumulation over
 *            head_dim, rounded once to nearest
 *
 * palu_output_proj is the per-step GEMV y = o W_fused on the current device:
 *   W_fused  device [k_dim][d_model] F16/BF16, 16-byte aligned; k_dim = n_heads * rank_v
 *   o        device [batch][k_dim] float32 (palu_decode_attn's `out`, [batch][n][rank_v])
 *   y        device [batch][d_model] float32, overwritten
 *   workspace device, 256-byte aligned, palu_output_proj_workspace_size(k_dim, d_model,
 *            max_batch) bytes for any batch <= max_batch; it must be zero-filled before
 *            its first use, and every call leaves it ready for the next. Calls sharing a
 *            workspace must not overlap on the GPU.
 * d_model must be a multiple of 8 (else PALU_ERR_INVALID_ARG); k_dim <= 65536 and
 * batch <= 1024 (else PALU_ERR_UNSUPPORTED). The result is deterministic (fixed
 * summation order).
 * `stream` must belong to the calling thread's current device (else
 * PALU_ERR_INVALID_ARG). Asynchronous on `stream`.
 */
palu_status_t palu_fuse_value_output(const void* B_v, const void* W_o, palu_dtype_t in_dtype, int n_heads,
                                     int head_dim, int group_size, int rank_v, int64_t d_model, void* W_fused,
                                     palu_dtype_t out_dtype, palu_stream_t stream);
palu_status_t palu_output_proj_workspace_size(int64_t k_dim, int64_t d_model, int max_batch, size_t* bytes);
palu_status_t palu_output_proj(const void* W_fused, palu_dtype_t w_dtype, int64_t k_dim, int64_t d_model,
                               const float* o, int batch, float* y, void* workspace, size_t workspace_bytes,
                               palu_stream_t stream);

/*
 * Decode over a hybrid cache: dense attention-sink and recent-window tokens kept as a standard
 * KV cache next to the G-LRD latent middle ("PuzzleKV" section 3: the sink page and the local
 * window stay dense, the other pages are factorised, and each query attends over both kinds of
 * page, the partial results merged by online softmax; "Shard" section 7: four fp16 sink tokens
 * and a 64-token fp16 window around the compressed middle).
 *
 *   dense->k, dense->v  device [max_rows][capacity][n_heads][head_dim] in dense->dtype (F32, F16
 *                       or BF16), 8-byte aligned for F16 / BF16 and 4-byte for F32 (else
 *                       PALU_ERR_INVALID_ARG). On the RoPE path the keys are stored rotated at their
 *                       own positions (as a dense KV cache holds them); on the absorbed path unrotated.
 *   dense->n_tokens     device [batch] int32: tokens 0 .. n_tokens[b] - 1 of row b are attended
 *                       (their order does not matter); a count outside [0, capacity] is clamped
 *                       and recorded in the error word.
 *
 * The other arguments are palu_decode_attn's, for the latent middle only: seq_lens counts its
 * tokens and `positions` gives their positions (the middle usually starts after the sink tokens,
 * so the default t is rarely right). q_pos is required on the RoPE path (the position of the
 * decoded token). lse is required. One softmax spans both segments; the outputs are
 *   out       [batch][n_heads][rank_v]    sum over the middle of p h_v (latent space)
 *   out_dense [batch][n_heads][head_dim]  sum over the dense tokens of p v (value space)
 *   lse       [batch][n_heads]            natural log-sum-exp over all tokens
 * so head i's attention output is out_i B_v^(i) + out_dense_i (out feeds palu_output_proj with
 * the fused weight, out_dense the plain W_o). Supported head_dim: 32, 64, 96 or 128 (else
 * PALU_ERR_UNSUPPORTED). Two launches on `stream`: the latent decode, then the dense merge.
 */
typedef struct palu_dense_cache {
  const void* k;
  const void* v;
  const int32_t* n_tokens;
  int64_t capacity;
  palu_dtype_t dtype;
} palu_dense_cache;

palu_status_t palu_decode_hybrid(palu_attn_t h, const void* q, const palu_cache* cache, const int32_t* seq_lens,
                                 const int32_t* positions, const int32_t* q_pos, int batch, int64_t max_seq_len,
                                 const palu_dense_cache* dense, float* out, float* out_dense, float* lse,
                                 palu_stream_t stream);

/*
 * Decode over a page-factorised cache ("PuzzleKV" section 3.3, eq. 2 and step 4): every completed
 * page of P tokens of a head stores its keys and values as rank-r factors, K_p ~= L_K R_K and
 * V_p ~= L_V R_V (L: P x r with orthonormal columns from the page's truncated SVD, R: r x d_h).
 * A page is scored as s = (q R_K^T) L_K^T / sqrt(d_h) and its values are read as p L_V R_V,
 * without rebuilding the page. The dense sink and window tokens, when given, share the softmax.
 * This is the PuzzleKV alternative to the G-LRD latent middle of palu_decode_hybrid; the handle
 * supplies the heads, head_dim, q dtype, mode, RoPE table and workspace (its latent shape is not
 * used).
 *
 *   pages->pages     device, 16-byte aligned: [max_rows][capacity][n_heads] page records, each
 *                    L_K [P][r], R_K [r][head_dim], L_V [P][r], R_V [r][head_dim] row-major and
 *                    contiguous (640 r bytes for P = 32, head_dim 128), in pages->dtype (F16/BF16).
 *                    On the RoPE path the factorised keys are the stored, rotated keys.
 *   pages->n_pages   device [batch] int32: pages 0 .. n_pages[b] - 1 of row b are attended; a
 *                    count outside [0, max_pages] is clamped and recorded in the error word.
 *   max_pages        bound on n_pages for this call (<= capacity); it sizes the split plan.
 *   dense            NULL, or the sink / window tokens as for palu_decode_hybrid.
 *   q                [batch][n_heads][head_dim] in the handle's q dtype, unrotated; q_pos [batch]
 *                    is required on the RoPE path.
 *   out              [batch][n_heads][head_dim]: sum over the pages of p (L_V R_V) (value space)
 *   out_dense        [batch][n_heads][head_dim] when dense is given: sum over the dense tokens
 *   lse              [batch][n_heads], required: natural log-sum-exp over all attended tokens
 * so the attention output is out + out_dense. Supported: head_dim 128, P = 32, r in {8, 16, 32}
 * (else PALU_ERR_UNSUPPORTED); PALU_FLAG_ALIBI handles are refused (no positions). The split partials
 * live in the handle's workspace; a handle too small for one head_dim-wide partial per (row, head)
 * (rank_v below head_dim with max_tokens <= 16) gives PALU_ERR_WORKSPACE. One launch, two with the
 * dense segment, asynchronous on `stream`.
 */
typedef struct palu_page_cache {
  const void* pages;
  const int32_t* n_pages;
  int64_t capacity;
  int page_size;
  int rank;
  palu_dtype_t dtype;
} palu_page_cache;

palu_status_t palu_decode_paged(palu_attn_t h, const void* q, const palu_page_cache* pages, const int32_t* q_pos,
                                int batch, int64_t max_pages, const palu_dense_cache* dense, float* out,
                                float* out_dense, float* lse, palu_stream_t stream);

/*
 * Latent production: the step that fills the cache ("方法细节", SVD-rewrite paragraph: the
 * layer caches h = x A in place of k = x W and v = x W_v; G-LRD paragraph: one A_g per group;
 * "补充细节": per-token quantisation of the cached latents). For n_new new tokens of each
 * batch row, H_k = x A_k,g and H_v = x A_v,g are computed on the tensor cores (fp16 or bf16
 * operands, fp32 accumulation) and written into the cache at tokens dst_slot[b] ..
 * dst_slot[b] + n_new - 1 of row b, in the cache's dtype: F32 values as accumulated, F16/BF16
 * rounded to nearest, INT4 quantised per token and group exactly as palu_append_latents does
 * (the same codes and scales for the same fp32 values).
 *
 * palu_down_proj_size / palu_prepare_down_proj (once per layer, an offline transform): A_k and
 * A_v are device arrays [n_g][d_model][rank] in a_dtype (F32, F16, BF16), the Hadamard-folded
 * factors where the latents are rotated. W (device, 16-byte aligned, palu_down_proj_size
 * bytes) receives [2][n_g][rank][d_model] in w_dtype (F16 or BF16): each A_g transposed.
 *
 * palu_project_latents (per prefill or decode step): x device [batch][n_new][d_model] in
 * w_dtype, 16-byte aligned; W as prepared; cache and dst_slot as for palu_append_latents.
 * Supported: rank_k = rank_v in {128, 256}, key and value caches of one dtype, d_model a
 * multiple of 64, batch * n_new < 2^31 (else PALU_ERR_UNSUPPORTED). A slot past the capacity
 * is recorded in the error word and that token's rows are skipped. Asynchronous on `stream`.
 */
palu_status_t palu_down_proj_size(palu_attn_t h, int64_t d_model, size_t* bytes);
palu_status_t palu_prepare_down_proj(palu_attn_t h, const void* A_k, const void* A_v, palu_dtype_t a_dtype,
                                     int64_t d_model, palu_dtype_t w_dtype, void* W, size_t W_bytes,
                                     palu_stream_t stream);
palu_status_t palu_project_latents(palu_attn_t h, const void* W, palu_dtype_t w_dtype, int64_t d_model,
                                   const void* x, const palu_cache* cache, const int32_t* dst_slot, int batch,
                                   int n_new, palu_stream_t stream);

/* Free the host handle. Does not synchronise: no work on it may be in flight. NULL is fine. */
palu_status_t palu_destroy(palu_attn_t h);

/* Read and clear the device error word (synchronises `stream`). PALU_OK if nothing was recorded. */
palu_status_t palu_attn_check(palu_attn_t h, palu_stream_t stream);

/*
 * Tracing. While enabled, every palu_decode_attn call records a pair of CUDA
 * events around its main attention kernel, on the call's stream, into a ring of
 * PALU_TRACE_CAPACITY pairs (the events are created by the library and hold no
 * device memory; launches beyond the capacity are not recorded).
 * palu_attn_trace_read waits for the recorded events, returns the number of
 * recorded launches and their summed device time in milliseconds, and empties
 * the ring. Disabling destroys the events.
 */
#define PALU_TRACE_CAPACITY 4096
palu_status_t palu_attn_trace_enable(palu_attn_t h, int enable);
palu_status_t palu_attn_trace_read(palu_attn_t h, int* launches, double* total_ms);
/*
 * Like palu_attn_trace_read, but writes each recorded launch's device time in
 * milliseconds, in launch order, to ms[0 .. launches) (host memory, `capacity`
 * entries; launches beyond it are dropped) and empties the ring.
 */
palu_status_t palu_attn_trace_times(palu_attn_t h, float* ms, int capacity, int* launches);

/* Static description of a status code. */
const char* palu_status_string(palu_status_t s);

/*
 * Test hook for the int4 load path of the CUDA-core kernel (PALU_KERNEL_SIMT, which
 * runs int4 absorbed decodes and the int4 shapes the tensor-core kernel does not
 * take): writes, as float32, the dequantised latents (code * scale) of tokens
 * [0, n_tokens) of cache rows [0, batch) into out [batch][n_tokens][n_g][rank]
 * (device), with that kernel's unpack routine. which = 0 for keys, 1 for values.
 * The tensor-core kernel unpacks with other routines; palu_debug_int4_operand and
 * palu_debug_int4_dp2a export those.
 */
palu_status_t palu_debug_dequant(palu_attn_t h, const palu_cache* cache, int which, int batch,
                                 int64_t n_tokens, float* out, palu_stream_t stream);

/*
 * Test hooks for the int4 path of the tensor-core RoPE kernel (PALU_KERNEL_TC_ROPE).
 * They run that kernel's own device routines, so that a bit-exact comparison checks
 * the code that decodes. The pages fix the stored format (per-token int4 latents,
 * "补充细节" KV-quantisation paragraph; codes in [-7, 7]); the routines are this
 * library's.
 *
 * palu_debug_int4_operand -- the key side. For every 128-token tile of rows [0, batch)
 * it loads the packed key codes into shared memory with the decode kernel's TMA
 * box and 128-byte swizzle, expands each token row with the decode kernel's
 * converter into the swizzled fp16 tensor-core operand, reads the operand back and
 * writes, for tokens [0, n_tokens):
 *   codes  device [batch][n_tokens][n_g][rank_k] uint16: the fp16 bit pattern of each
 *          operand element (the signed code as an exact fp16 number), in the operand's
 *          rank order: within every run of eight consecutive ranks, position p holds
 *          rank {0, 2, 4, 6, 1, 3, 5, 7}[p] (B_k^T is stored with the same order)
 *   deq    device float, same shape and order: operand value x the token's key scale
 *          (exact in fp32), or NULL
 * Requires desc.k_dtype = PALU_INT4 and rank_k = 256 (else PALU_ERR_INVALID_ARG /
 * PALU_ERR_UNSUPPORTED) and batch * capacity >= 128 (else PALU_ERR_UNSUPPORTED). A
 * bounded wait that gives up is reported by palu_attn_check as PALU_ERR_TIMEOUT.
 *
 * palu_debug_int4_dp2a -- the value side (which = 1; which = 0 runs the same routine
 * on the key codes). For every block of 16 tokens (tokens 16 k .. 16 k + 15 of
 * [0, n_tokens), missing tokens counting as weight 0) and both heads h = 0, 1 of a
 * head pair, the decode kernel's dp2a routine forms the exact integer sums
 *   sums[b][k][g][h][c] = sum_t weights[b][t][h] * code[b][t][g][c]
 * with weights device [batch][n_tokens][2] int32, each in [0, 32767] (the 15-bit
 * weights the decode kernel feeds it; other values give undefined sums), and
 * sums device [batch][ceil(n_tokens / 16)][n_g][2][rank] int32. Requires rank 256.
 */
palu_status_t palu_debug_int4_operand(palu_attn_t h, const palu_cache* cache, int batch, int64_t n_tokens,
                                      uint16_t* codes, float* deq, palu_stream_t stream);
palu_status_t palu_debug_int4_dp2a(palu_attn_t h, const palu_cache* cache, int which, int batch, int64_t n_tokens,
                                   const int32_t* weights, int32_t* sums, palu_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PALU_ATTN_H */
