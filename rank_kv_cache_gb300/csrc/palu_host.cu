// C ABI of the G-LRD decode-attention library: validation, workspace layout,
// launch planning and dispatch. Host code only; kernels live in the other units.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "palu_attn.h"
#include "internal.h"

using namespace palu;

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int elem_bytes(palu_dtype_t t) { return t == PALU_F32 ? 4 : 2; }

struct WsLayout {
  size_t err, bk, bkt, rope, phase, qbuf, part_o, part_ml, counters, total;
  int max_splits;
  int64_t max_pos;
};

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

palu_status_t check_desc(const palu_attn_desc* d) {
  if (!d) return PALU_ERR_INVALID_ARG;
  if (d->abi_version != PALU_ABI_VERSION) return PALU_ERR_INVALID_ARG;
  if (d->n_heads <= 0 || d->group_size <= 0 || d->n_heads % d->group_size != 0) return PALU_ERR_INVALID_ARG;
  if (d->max_batch <= 0 || d->max_tokens <= 0 || d->max_position < 0) return PALU_ERR_INVALID_ARG;
  if (d->max_tokens > (int64_t)1 << 30 || d->max_position > (int64_t)1 << 30) return PALU_ERR_INVALID_ARG;
  if ((d->flags & ~(PALU_FLAG_TEST_STALL | PALU_FLAG_ALIBI)) != 0) return PALU_ERR_INVALID_ARG;
  if (d->mode != PALU_MODE_ROPE && d->mode != PALU_MODE_ABSORBED) return PALU_ERR_INVALID_ARG;
  if ((d->flags & PALU_FLAG_ALIBI) && d->mode != PALU_MODE_ABSORBED) return PALU_ERR_INVALID_ARG;
  if ((unsigned)d->k_dtype > PALU_INT4 || (unsigned)d->v_dtype > PALU_INT4) return PALU_ERR_INVALID_ARG;
  if ((unsigned)d->bk_dtype > PALU_BF16 || (unsigned)d->q_dtype > PALU_BF16) return PALU_ERR_INVALID_ARG;
  if (d->mode == PALU_MODE_ROPE && !(d->rope_theta > 0.0 && isfinite(d->rope_theta))) return PALU_ERR_INVALID_ARG;
  if (d->head_dim <= 0 || d->rank_k <= 0 || d->rank_v <= 0) return PALU_ERR_INVALID_ARG;
  // shapes and type combinations with a kernel in this build
  if (d->head_dim != 64 && d->head_dim != 128) return PALU_ERR_UNSUPPORTED;
  // group sizes 1..8 run on every path; 16 and 32 (joint decomposition of up to all 32 heads of a
  // Llama-2-7B layer) only on the tensor-core RoPE kernel, whose shape rules they must meet
  const bool tc_shape = d->mode == PALU_MODE_ROPE && d->head_dim == 128 && d->rank_k == 256 && d->rank_v == 256 &&
                        (d->k_dtype == PALU_F16 || d->k_dtype == PALU_BF16 || d->k_dtype == PALU_INT4);
  // ... and on the absorbed path as split groups (rank 256, fp16 / bf16 latents)
  const bool split_shape = d->mode == PALU_MODE_ABSORBED && d->rank_k == 256 && d->rank_v == 256 &&
                           d->k_dtype == d->v_dtype && (d->k_dtype == PALU_F16 || d->k_dtype == PALU_BF16);
  if (!pow2_in(d->group_size, 1, 8) && !((tc_shape || split_shape) && (d->group_size == 16 || d->group_size == 32)))
    return PALU_ERR_UNSUPPORTED;
  if (!pow2_in(d->rank_k, 64, 256) || !pow2_in(d->rank_v, 64, 256)) return PALU_ERR_UNSUPPORTED;
  // one latent dtype for keys and values, or int4 values under fp16 / bf16 keys (V-only int4)
  if (d->v_dtype != d->k_dtype && !(d->v_dtype == PALU_INT4 && (d->k_dtype == PALU_F16 || d->k_dtype == PALU_BF16)))
    return PALU_ERR_UNSUPPORTED;
  const palu_dtype_t want_bk = d->k_dtype == PALU_INT4 ? PALU_F16 : d->k_dtype;
  if (d->bk_dtype != want_bk) return PALU_ERR_UNSUPPORTED;
  return PALU_OK;
}

// The group shape the decode kernels run. G-LRD groups of s = 1 (M-LRD) or s = 2 heads with
// r = 64 s ranks each, fp16 or bf16 latents and d_h = 128, are run as groups of four heads and
// 256 ranks: 4 / s neighbouring groups' cache rows are contiguous, so the cache is read as is, and
// their B_k blocks form a block-diagonal B_k of the packed group (zeros elsewhere). A head's
// scores then equal its own group's exactly (the other groups' latents meet zeros); its output
// is the slice of the packed group's 256 latent columns that holds its own group's ranks, which
// the split merge writes. This puts those shapes on the tensor-core and TMA-streamed kernels.
// On the absorbed path, groups of 8, 16 or 32 heads at 256 ranks (fp16/bf16) are split the other
// way: each runs as s / 4 kernel groups of four heads that read the same cache group, each with its
// own column block of B_k, so the TMA-streamed kernel (four heads per CTA) takes them too.
struct KShape {
  int s, rk, rv, pack;   // pack = source groups per kernel group (1: none)
  int split;             // kernel groups per source group (1: none)
  int64_t n_g;
};

KShape kernel_shape(const palu_attn_desc& d) {
  KShape k{d.group_size, d.rank_k, d.rank_v, 1, 1, d.n_heads / d.group_size};
  if (d.mode == PALU_MODE_ABSORBED && (d.group_size == 8 || d.group_size == 16 || d.group_size == 32) &&
      d.rank_k == 256 && d.rank_v == 256 && d.k_dtype == d.v_dtype && (d.k_dtype == PALU_F16 || d.k_dtype == PALU_BF16)) {
    k.split = d.group_size / 4;
    k.s = 4;
    k.n_g = d.n_heads / 4;
    return k;
  }
  if ((d.group_size == 1 || d.group_size == 2) && d.head_dim == 128 && d.rank_k == 64 * d.group_size &&
      d.rank_v == d.rank_k && d.n_heads % 4 == 0 && d.k_dtype == d.v_dtype &&
      (d.k_dtype == PALU_F16 || d.k_dtype == PALU_BF16)) {
    k.pack = 4 / d.group_size;
    k.s = 4;
    k.rk = k.rv = 256;
    k.n_g = d.n_heads / 4;
  }
  return k;
}

WsLayout layout_of(const palu_attn_desc& d) {
  WsLayout L{};
  const KShape k = kernel_shape(d);
  const int64_t n_g = k.n_g;
  const int64_t cols = (int64_t)k.s * d.head_dim;
  L.max_pos = d.max_position > 0 ? d.max_position : d.max_tokens;
  int64_t ms = (d.max_tokens + kSimtTile - 1) / kSimtTile;
  L.max_splits = int(ms < 1 ? 1 : (ms > 256 ? 256 : ms));
  size_t off = 0;
  L.err = off;
  off = align256(off + 256);
  L.bk = off;
  off = align256(off + (size_t)n_g * k.rk * cols * elem_bytes(d.bk_dtype));
  L.bkt = off;
  if (d.mode == PALU_MODE_ROPE && d.k_dtype != PALU_F32) off = align256(off + (size_t)n_g * cols * k.rk * 2);
  L.rope = off;
  if (d.mode == PALU_MODE_ROPE) off = align256(off + (size_t)L.max_pos * (d.head_dim / 2) * sizeof(float2));
  L.phase = off;
  if (d.mode == PALU_MODE_ROPE) off = align256(off + (size_t)(d.head_dim / 2) * sizeof(uint64_t));
  const int qw = d.mode == PALU_MODE_ROPE ? d.head_dim : k.rk;
  L.qbuf = off;
  off = align256(off + (size_t)d.max_batch * d.n_heads * qw * sizeof(float));
  L.part_o = off;
  off = align256(off + (size_t)d.max_batch * d.n_heads * L.max_splits * k.rv * sizeof(float));
  L.part_ml = off;
  off = align256(off + (size_t)d.max_batch * d.n_heads * L.max_splits * sizeof(float2));
  L.counters = off;
  off = align256(off + (size_t)d.max_batch * d.n_heads * sizeof(unsigned));
  L.total = off;
  return L;
}

int to_dt(palu_dtype_t t) { return (int)t; }

// Split-T plan. `slots` CTAs run at once; each unit (one CTA's share of a group) is cut
// into `splits` ranges of `tps` tiles. Picks the split count with the smallest estimated
// time waves * (tps + fixed), where `fixed` is a CTA's fixed cost in tiles (prologue operand
// loads, pipeline fill and drain, partial write and merge), which also keeps splits from
// growing without need.
void plan_splits(int64_t tiles, int64_t units, int64_t slots, int64_t max_splits, int fixed, int* n_splits,
                 int* tps_out) {
  int64_t cap = tiles < max_splits ? tiles : max_splits;
  if (cap < 1) cap = 1;
  double best = 1e300;
  int64_t best_s = 1, best_t = tiles;
  for (int64_t s = 1; s <= cap; ++s) {
    const int64_t tps = (tiles + s - 1) / s;
    const int64_t s2 = (tiles + tps - 1) / tps;
    if (s2 != s) continue;  // same plan as a smaller split count
    const int64_t waves = (units * s2 + slots - 1) / slots;
    const double est = double(waves) * double(tps + fixed);
    if (est < best - 1e-9) {
      best = est;
      best_s = s2;
      best_t = tps;
    }
  }
  *n_splits = (int)best_s;
  *tps_out = (int)best_t;
}

}  // namespace

struct Trace {
  bool on = false;
  int n = 0;                       // recorded pairs
  int created = 0;                 // events created so far (pairs)
  cudaEvent_t ev[2 * PALU_TRACE_CAPACITY];
};

struct palu_attn {
  palu_attn_desc d;
  Trace trace;
  char* ws;
  size_t ws_bytes;
  WsLayout L;
  int n_g;       // groups of the descriptor (cache rows, append, latent production)
  KShape ks;     // the group shape the decode kernels run
  int device;
  int sm_count;
  int mma_dtype;
};

extern "C" {

const char* palu_status_string(palu_status_t s) {
  switch (s) {
    case PALU_OK: return "ok";
    case PALU_ERR_INVALID_ARG: return "invalid argument";
    case PALU_ERR_UNSUPPORTED: return "unsupported shape or dtype combination";
    case PALU_ERR_CUDA: return "CUDA runtime error";
    case PALU_ERR_DEVICE: return "a kernel recorded an out-of-range index";
    case PALU_ERR_TIMEOUT: return "a bounded device wait gave up";
    case PALU_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

palu_status_t palu_attn_workspace_size(const palu_attn_desc* desc, size_t* bytes) {
  if (!bytes) return PALU_ERR_INVALID_ARG;
  const palu_status_t st = check_desc(desc);
  if (st != PALU_OK) return st;
  *bytes = layout_of(*desc).total;
  return PALU_OK;
}

palu_status_t palu_attn_create(const palu_attn_desc* desc, const void* B_k, void* workspace, size_t workspace_bytes,
                               palu_stream_t stream, palu_attn_t* out) {
  if (!out) return PALU_ERR_INVALID_ARG;
  *out = nullptr;
  palu_status_t st = check_desc(desc);
  if (st != PALU_OK) return st;
  if (!B_k) return PALU_ERR_INVALID_ARG;
  if ((uintptr_t)B_k % 16) return PALU_ERR_INVALID_ARG;
  const WsLayout L = layout_of(*desc);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < L.total) return PALU_ERR_WORKSPACE;

  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, workspace) != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return PALU_ERR_WORKSPACE;
  }
  if (cudaSetDevice(attr.device) != cudaSuccess) return PALU_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, attr.device) != cudaSuccess) return PALU_ERR_CUDA;

  palu_attn* h = new (std::nothrow) palu_attn();
  if (!h) return PALU_ERR_INVALID_ARG;
  h->d = *desc;
  h->ws = static_cast<char*>(workspace);
  h->ws_bytes = workspace_bytes;
  h->L = L;
  h->n_g = desc->n_heads / desc->group_size;
  h->ks = kernel_shape(*desc);
  h->device = attr.device;
  h->sm_count = sms;
  h->mma_dtype = desc->k_dtype == PALU_BF16 ? kBF16 : kF16;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(h->ws + L.err, 0, 256, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(h->ws + L.counters, 0, (size_t)desc->max_batch * desc->n_heads * sizeof(unsigned), s);
  const KShape& k = h->ks;
  void* bkt = (desc->mode == PALU_MODE_ROPE && desc->k_dtype != PALU_F32) ? h->ws + L.bkt : nullptr;
  if (e == cudaSuccess)
    e = launch_copy_bk(B_k, to_dt(desc->bk_dtype), h->ws + L.bk, bkt, h->mma_dtype, (int)k.n_g, k.rk,
                       k.s * desc->head_dim, desc->head_dim, desc->k_dtype == PALU_INT4 ? 1 : 0, k.pack, k.split,
                       desc->group_size, desc->rank_k, s);
  if (e == cudaSuccess && desc->mode == PALU_MODE_ROPE)
    e = launch_rope_table(reinterpret_cast<float2*>(h->ws + L.rope), reinterpret_cast<uint64_t*>(h->ws + L.phase),
                          L.max_pos, desc->head_dim, desc->rope_theta, s);
  if (e != cudaSuccess) {
    delete h;
    return PALU_ERR_CUDA;
  }
  *out = h;
  return PALU_OK;
}

static void trace_destroy(palu_attn* h) {
  for (int i = 0; i < 2 * h->trace.created; ++i) cudaEventDestroy(h->trace.ev[i]);
  h->trace.created = 0;
  h->trace.n = 0;
}

palu_status_t palu_destroy(palu_attn_t h) {
  if (!h) return PALU_OK;
  if (h->trace.created) {
    cudaSetDevice(h->device);
    trace_destroy(h);
  }
  delete h;
  return PALU_OK;
}

palu_status_t palu_attn_trace_enable(palu_attn_t h, int enable) {
  if (!h) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  if (!enable) trace_destroy(h);
  h->trace.on = enable != 0;
  h->trace.n = 0;
  return PALU_OK;
}

palu_status_t palu_attn_trace_read(palu_attn_t h, int* launches, double* total_ms) {
  if (!h || !launches || !total_ms) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  double sum = 0.0;
  for (int i = 0; i < h->trace.n; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(h->trace.ev[2 * i + 1]) != cudaSuccess) return PALU_ERR_CUDA;
    if (cudaEventElapsedTime(&ms, h->trace.ev[2 * i], h->trace.ev[2 * i + 1]) != cudaSuccess) return PALU_ERR_CUDA;
    sum += ms;
  }
  *launches = h->trace.n;
  *total_ms = sum;
  h->trace.n = 0;
  return PALU_OK;
}

palu_status_t palu_attn_trace_times(palu_attn_t h, float* ms, int capacity, int* launches) {
  if (!h || !launches || capacity < 0 || (capacity > 0 && !ms)) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const int n = h->trace.n < capacity ? h->trace.n : capacity;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(h->trace.ev[2 * i + 1]) != cudaSuccess) return PALU_ERR_CUDA;
    if (cudaEventElapsedTime(&ms[i], h->trace.ev[2 * i], h->trace.ev[2 * i + 1]) != cudaSuccess) return PALU_ERR_CUDA;
  }
  *launches = n;
  h->trace.n = 0;
  return PALU_OK;
}

// Event pair for the next traced launch, or nullptr when tracing is off or the ring is full.
static cudaEvent_t* trace_slot(palu_attn* h) {
  Trace& t = h->trace;
  if (!t.on || t.n >= PALU_TRACE_CAPACITY) return nullptr;
  if (t.n >= t.created) {
    if (cudaEventCreate(&t.ev[2 * t.n]) != cudaSuccess) return nullptr;
    if (cudaEventCreate(&t.ev[2 * t.n + 1]) != cudaSuccess) {
      cudaEventDestroy(t.ev[2 * t.n]);
      return nullptr;
    }
    t.created = t.n + 1;
  }
  return &t.ev[2 * t.n++];
}

palu_status_t palu_attn_check(palu_attn_t h, palu_stream_t stream) {
  if (!h) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ErrWord w{};
  if (cudaMemcpyAsync(&w, h->ws + h->L.err, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PALU_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PALU_ERR_CUDA;
  if (w.code == 0) return PALU_OK;
  if (cudaMemsetAsync(h->ws + h->L.err, 0, sizeof(w), s) != cudaSuccess) return PALU_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PALU_ERR_CUDA;
  return w.code == kCodeTimeout ? PALU_ERR_TIMEOUT : PALU_ERR_DEVICE;
}

static palu_status_t check_cache(const palu_attn* h, const palu_cache* c) {
  if (!c || !c->hk || !c->hv || c->capacity <= 0) return PALU_ERR_INVALID_ARG;
  if ((uintptr_t)c->hk % 16 || (uintptr_t)c->hv % 16) return PALU_ERR_INVALID_ARG;
  if (h->d.k_dtype == PALU_INT4 && (!c->k_scale || (uintptr_t)c->k_scale % 2)) return PALU_ERR_INVALID_ARG;
  if (h->d.v_dtype == PALU_INT4 && (!c->v_scale || (uintptr_t)c->v_scale % 2)) return PALU_ERR_INVALID_ARG;
  return PALU_OK;
}

palu_status_t palu_append_latents(palu_attn_t h, const palu_cache* cache, const void* hk_new, const void* hv_new,
                                  palu_dtype_t src_dtype, const int32_t* dst_slot, int batch, int n_new,
                                  palu_stream_t stream) {
  if (!h) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  if (batch < 0 || batch > h->d.max_batch || n_new < 0) return PALU_ERR_INVALID_ARG;
  if ((unsigned)src_dtype > PALU_BF16) return PALU_ERR_INVALID_ARG;
  if (batch == 0 || n_new == 0) return PALU_OK;
  if (!hk_new || !hv_new || !dst_slot) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ErrWord* err = reinterpret_cast<ErrWord*>(h->ws + h->L.err);
  const cudaError_t e = launch_append(cache->hk, static_cast<__half*>(cache->k_scale), h->d.rank_k, hk_new,
                                      cache->hv, static_cast<__half*>(cache->v_scale), h->d.rank_v, hv_new,
                                      to_dt(h->d.k_dtype), to_dt(h->d.v_dtype), cache->capacity, h->n_g,
                                      to_dt(src_dtype), dst_slot, batch, n_new, err, s);
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

// ---------------------------------------------------------------------------- latent production
// The prepared down-projection operand is [2][n_g][rank][d_model] (A_k then A_v, each A_g
// transposed); the tensor-core kernel takes rank 128 or 256 and d_model in multiples of 64.
static palu_status_t check_down_proj(const palu_attn* h, int64_t d_model) {
  if (!h || d_model <= 0) return PALU_ERR_INVALID_ARG;
  if (h->d.rank_k != h->d.rank_v || (h->d.rank_k != 128 && h->d.rank_k != 256) || d_model % 64 ||
      d_model > (int64_t(1) << 31))
    return PALU_ERR_UNSUPPORTED;
  return PALU_OK;
}

palu_status_t palu_down_proj_size(palu_attn_t h, int64_t d_model, size_t* bytes) {
  if (!bytes) return PALU_ERR_INVALID_ARG;
  const palu_status_t st = check_down_proj(h, d_model);
  if (st != PALU_OK) return st;
  *bytes = (size_t)2 * h->n_g * h->d.rank_k * d_model * 2;
  return PALU_OK;
}

palu_status_t palu_prepare_down_proj(palu_attn_t h, const void* A_k, const void* A_v, palu_dtype_t a_dtype,
                                     int64_t d_model, palu_dtype_t w_dtype, void* W, size_t W_bytes,
                                     palu_stream_t stream) {
  palu_status_t st = check_down_proj(h, d_model);
  if (st != PALU_OK) return st;
  if ((unsigned)a_dtype > PALU_BF16 || (w_dtype != PALU_F16 && w_dtype != PALU_BF16)) return PALU_ERR_INVALID_ARG;
  const size_t ie = a_dtype == PALU_F32 ? 4 : 2;
  if (!A_k || !A_v || !W || (uintptr_t)A_k % ie || (uintptr_t)A_v % ie || (uintptr_t)W % 16) return PALU_ERR_INVALID_ARG;
  if (W_bytes < (size_t)2 * h->n_g * h->d.rank_k * d_model * 2) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const cudaError_t e = launch_prepare_down_proj(A_k, A_v, to_dt(a_dtype), h->n_g, h->d.rank_k, d_model,
                                                 to_dt(w_dtype), W, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

palu_status_t palu_project_latents(palu_attn_t h, const void* W, palu_dtype_t w_dtype, int64_t d_model,
                                   const void* x, const palu_cache* cache, const int32_t* dst_slot, int batch,
                                   int n_new, palu_stream_t stream) {
  palu_status_t st = check_down_proj(h, d_model);
  if (st != PALU_OK) return st;
  st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  if (h->d.k_dtype != h->d.v_dtype) return PALU_ERR_UNSUPPORTED;
  if (w_dtype != PALU_F16 && w_dtype != PALU_BF16) return PALU_ERR_INVALID_ARG;
  if (batch < 0 || batch > h->d.max_batch || n_new < 0) return PALU_ERR_INVALID_ARG;
  if ((int64_t)batch * n_new >= (int64_t(1) << 31)) return PALU_ERR_UNSUPPORTED;
  if (batch == 0 || n_new == 0) return PALU_OK;
  if (!W || !x || !dst_slot || (uintptr_t)W % 16 || (uintptr_t)x % 16) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  ProjectArgs a{};
  a.cache[0] = cache->hk;
  a.cache[1] = cache->hv;
  a.scale[0] = static_cast<__half*>(cache->k_scale);
  a.scale[1] = static_cast<__half*>(cache->v_scale);
  a.cache_dtype = to_dt(h->d.k_dtype);
  a.capacity = cache->capacity;
  a.n_g = h->n_g;
  a.rank = h->d.rank_k;
  a.d = d_model;
  a.dst_slot = dst_slot;
  a.n_new = n_new;
  a.M = (int64_t)batch * n_new;
  a.err = reinterpret_cast<ErrWord*>(h->ws + h->L.err);
  a.wait_ns = 1000000000ull;
  const cudaError_t e = launch_project_latents(x, W, w_dtype == PALU_BF16, a, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PALU_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

// Shape, type and workspace fields of a decode launch (the per-call pointers are set by the caller).
static void fill_args(const palu_attn* h, const palu_cache* cache, int batch, int64_t max_seq_len, DecodeArgs& a) {
  const palu_attn_desc& d = h->d;
  a.hk = cache->hk;
  a.hv = cache->hv;
  a.k_scale = static_cast<const __half*>(cache->k_scale);
  a.v_scale = static_cast<const __half*>(cache->v_scale);
  a.capacity = cache->capacity;
  a.n_heads = d.n_heads;
  a.n_g = (int)h->ks.n_g;
  a.s = h->ks.s;
  a.dh = d.head_dim;
  a.rk = h->ks.rk;
  a.rv = h->ks.rv;
  a.out_rv = h->ks.pack > 1 ? d.rank_v : 0;   // packed groups: the merge writes each head's own slice
  a.pack_s = d.group_size;
  a.g_split = h->ks.split;
  a.k_dtype = to_dt(d.k_dtype);
  a.v_dtype = to_dt(d.v_dtype);
  a.bk_dtype = to_dt(d.bk_dtype);
  a.batch = batch;
  a.max_seq_len = (int)max_seq_len;
  a.max_pos = h->L.max_pos;
  a.qbuf = reinterpret_cast<const float*>(h->ws + h->L.qbuf);
  a.bk = h->ws + h->L.bk;
  a.bkt = h->ws + h->L.bkt;
  a.rope = reinterpret_cast<const float2*>(h->ws + h->L.rope);
  a.phase = reinterpret_cast<const uint64_t*>(h->ws + h->L.phase);
  a.q_dtype = to_dt(d.q_dtype);
  a.qscale = float(1.4426950408889634 / sqrt((double)d.head_dim));
  a.part_o = reinterpret_cast<float*>(h->ws + h->L.part_o);
  a.part_ml = reinterpret_cast<float2*>(h->ws + h->L.part_ml);
  a.err = reinterpret_cast<ErrWord*>(h->ws + h->L.err);
  a.counters = reinterpret_cast<unsigned*>(h->ws + h->L.counters);  // the decode kernels merge the splits
  a.test_stall = (d.flags & PALU_FLAG_TEST_STALL) ? 1 : 0;
  a.alibi = (d.flags & PALU_FLAG_ALIBI) ? 1 : 0;
  a.wait_ns = a.test_stall ? 50000000ull : 1000000000ull;   // bound of every device wait
}

// Kernel choice and split-T plan: tensor-core rebuild (RoPE; fp16, bf16 and int4 latents),
// TMA stream (absorbed, fp16/bf16), CUDA-core kernel for everything else (fp32 latents, int4
// absorbed, other shapes). Sets a.n_splits / a.tiles_per_split; returns a palu_kernel_t.
static int plan_decode(const palu_attn* h, DecodeArgs& a) {
  const bool rope = h->d.mode == PALU_MODE_ROPE;
  const int kernel = (rope && tc_supported(a)) ? PALU_KERNEL_TC_ROPE
                     : (!rope && abs_supported(a)) ? PALU_KERNEL_TMA_ABSORBED
                                                   : PALU_KERNEL_SIMT;
  const int tile = kernel == PALU_KERNEL_TC_ROPE ? tc_tile_tokens()
                   : kernel == PALU_KERNEL_TMA_ABSORBED ? abs_stage_tokens()
                                                        : kSimtTile;
  const int64_t tiles = a.max_seq_len > 0 ? (a.max_seq_len + tile - 1) / tile : 1;
  const int64_t units = (int64_t)a.batch * a.n_g * (kernel == PALU_KERNEL_TC_ROPE ? tc_ctas_per_group(a) : 1);
  // CTA fixed costs in tiles, as measured on GB300 at the 32K-64K workloads: about four
  // 128-token tiles for the tensor-core kernel, eight 64-token stages for the absorbed stream
  const int fixed = kernel == PALU_KERNEL_TC_ROPE ? 4 : kernel == PALU_KERNEL_TMA_ABSORBED ? 8 : 1;
  plan_splits(tiles, units, kernel == PALU_KERNEL_SIMT ? 2 * h->sm_count : h->sm_count, h->L.max_splits, fixed,
              &a.n_splits, &a.tiles_per_split);
  return kernel;
}

palu_status_t palu_decode_plan(palu_attn_t h, int64_t cache_capacity, int batch, int64_t max_seq_len, int* kernel,
                               int* n_splits, int* launches) {
  if (!h || !kernel || !n_splits || !launches) return PALU_ERR_INVALID_ARG;
  if (cache_capacity <= 0 || batch <= 0 || batch > h->d.max_batch) return PALU_ERR_INVALID_ARG;
  if (max_seq_len < 0 || max_seq_len > h->d.max_tokens || max_seq_len > cache_capacity) return PALU_ERR_INVALID_ARG;
  palu_cache c{};
  c.capacity = cache_capacity;
  DecodeArgs a{};
  fill_args(h, &c, batch, max_seq_len, a);
  *kernel = plan_decode(h, a);
  *n_splits = a.n_splits;
  *launches = *kernel == PALU_KERNEL_TC_ROPE ? 1 : 2;  // the other kernels read a prepared query
  return PALU_OK;
}

palu_status_t palu_decode_attn(palu_attn_t h, const void* q, const palu_cache* cache, const int32_t* seq_lens,
                               const int32_t* positions, const int32_t* q_pos, int batch, int64_t max_seq_len,
                               float* out, float* lse, palu_stream_t stream) {
  if (!h) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  if (batch < 0 || batch > h->d.max_batch) return PALU_ERR_INVALID_ARG;
  if (batch == 0) return PALU_OK;
  if (!q || !seq_lens || !out) return PALU_ERR_INVALID_ARG;
  if ((uintptr_t)out % 16 || (uintptr_t)q % 4) return PALU_ERR_INVALID_ARG;
  if (max_seq_len < 0 || max_seq_len > h->d.max_tokens || max_seq_len > cache->capacity)
    return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  DecodeArgs a{};
  fill_args(h, cache, batch, max_seq_len, a);
  a.seq_lens = seq_lens;
  a.positions = (h->d.mode == PALU_MODE_ROPE || (h->d.flags & PALU_FLAG_ALIBI)) ? positions : nullptr;
  a.q = q;
  a.q_pos = q_pos;
  a.out = out;
  a.lse = lse;
  const int mode = h->d.mode == PALU_MODE_ROPE ? kRope : kAbsorbed;
  const int kernel = plan_decode(h, a);
  const bool use_tc = kernel == PALU_KERNEL_TC_ROPE, use_abs = kernel == PALU_KERNEL_TMA_ABSORBED;
  // group sizes above 8 have no CUDA-core kernel (a cache of fewer than 128 rows in all)
  if (kernel == PALU_KERNEL_SIMT && h->ks.s > 8) return PALU_ERR_UNSUPPORTED;

  // the tensor-core kernel rotates its query itself; the other kernels read the prepared buffer
  cudaError_t e = use_tc ? cudaSuccess
                         : launch_qprep(mode, q, a.q_dtype, a, q_pos, a.qscale, const_cast<float*>(a.qbuf), s);
  cudaEvent_t* tr = (e == cudaSuccess) ? trace_slot(h) : nullptr;
  if (tr) e = cudaEventRecord(tr[0], s);
  if (e == cudaSuccess)
    e = use_tc ? launch_decode_tc(a, s) : use_abs ? launch_decode_abs(a, s) : launch_decode_simt(mode, a, s);
  if (tr && e == cudaSuccess) e = cudaEventRecord(tr[1], s);
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

// Dense sink / window segment of a hybrid call merged into `out` (the other segment's output and
// lse), shared by palu_decode_hybrid's latent middle and palu_decode_paged's factorised pages.
static palu_status_t merge_dense_segment(const palu_attn* h, const DecodeArgs& a, const palu_dense_cache* dense,
                                         int batch, int out_width, const void* q, const int32_t* q_pos, float* out,
                                         float* out_dense, float* lse, palu_stream_t stream) {
  DenseArgs d{};
  d.k = dense->k;
  d.v = dense->v;
  d.dtype = to_dt(dense->dtype);
  d.n_tokens = dense->n_tokens;
  d.capacity = dense->capacity;
  d.n_heads = h->d.n_heads;
  d.dh = h->d.head_dim;
  d.rv = out_width;
  d.batch = batch;
  d.rope = h->d.mode == PALU_MODE_ROPE;
  d.q_pos = q_pos;
  d.rope_tab = a.rope;
  d.max_pos = a.max_pos;
  d.q = q;
  d.q_dtype = a.q_dtype;
  d.qscale = a.qscale;
  d.out = out;
  d.out_dense = out_dense;
  d.lse = lse;
  d.err = a.err;
  const cudaError_t e = launch_merge_dense(d, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

static palu_status_t check_dense(const palu_dense_cache* dense) {
  if (!dense->k || !dense->v || !dense->n_tokens || dense->capacity <= 0 || dense->capacity > (int64_t(1) << 31) ||
      (unsigned)dense->dtype > PALU_BF16)
    return PALU_ERR_INVALID_ARG;
  // 16-bit rows are read four elements (8 bytes) at a time
  const size_t al = dense->dtype == PALU_F32 ? 4 : 8;
  if ((uintptr_t)dense->k % al || (uintptr_t)dense->v % al) return PALU_ERR_INVALID_ARG;
  return PALU_OK;
}

palu_status_t palu_decode_hybrid(palu_attn_t h, const void* q, const palu_cache* cache, const int32_t* seq_lens,
                                 const int32_t* positions, const int32_t* q_pos, int batch, int64_t max_seq_len,
                                 const palu_dense_cache* dense, float* out, float* out_dense, float* lse,
                                 palu_stream_t stream) {
  if (!h || !dense) return PALU_ERR_INVALID_ARG;
  if (h->d.flags & PALU_FLAG_ALIBI) return PALU_ERR_UNSUPPORTED;   // the dense tokens carry no positions
  if (h->d.head_dim > 128 || h->d.head_dim % 32) return PALU_ERR_UNSUPPORTED;
  if (batch < 0 || batch > h->d.max_batch) return PALU_ERR_INVALID_ARG;
  if (batch == 0) return PALU_OK;
  if (!lse || !out_dense || (uintptr_t)out_dense % 4 || (uintptr_t)lse % 4) return PALU_ERR_INVALID_ARG;
  if (h->d.mode == PALU_MODE_ROPE && !q_pos) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_dense(dense);
  if (st != PALU_OK) return st;
  // the latent middle: out and lse hold its own softmax until the merge below
  st = palu_decode_attn(h, q, cache, seq_lens, positions, q_pos, batch, max_seq_len, out, lse, stream);
  if (st != PALU_OK) return st;
  DecodeArgs a{};
  fill_args(h, cache, batch, max_seq_len, a);
  return merge_dense_segment(h, a, dense, batch, h->d.rank_v, q, q_pos, out, out_dense, lse, stream);
}

palu_status_t palu_decode_paged(palu_attn_t h, const void* q, const palu_page_cache* pages, const int32_t* q_pos,
                                int batch, int64_t max_pages, const palu_dense_cache* dense, float* out,
                                float* out_dense, float* lse, palu_stream_t stream) {
  if (!h || !pages) return PALU_ERR_INVALID_ARG;
  if (h->d.flags & PALU_FLAG_ALIBI) return PALU_ERR_UNSUPPORTED;   // the pages carry no positions
  if (h->d.head_dim != 128) return PALU_ERR_UNSUPPORTED;
  if (pages->page_size != 32 || (pages->rank != 8 && pages->rank != 16 && pages->rank != 32) ||
      (pages->dtype != PALU_F16 && pages->dtype != PALU_BF16))
    return PALU_ERR_UNSUPPORTED;
  if (batch < 0 || batch > h->d.max_batch) return PALU_ERR_INVALID_ARG;
  if (batch == 0) return PALU_OK;
  if (!q || (uintptr_t)q % 4 || !out || (uintptr_t)out % 4 || !lse || (uintptr_t)lse % 4) return PALU_ERR_INVALID_ARG;
  if (!pages->pages || (uintptr_t)pages->pages % 16 || !pages->n_pages || pages->capacity <= 0) return PALU_ERR_INVALID_ARG;
  if (max_pages < 0 || max_pages > pages->capacity || max_pages > (int64_t(1) << 30)) return PALU_ERR_INVALID_ARG;
  if (h->d.mode == PALU_MODE_ROPE && !q_pos) return PALU_ERR_INVALID_ARG;
  if (dense) {
    const palu_status_t st = check_dense(dense);
    if (st != PALU_OK) return st;
    if (!out_dense || (uintptr_t)out_dense % 4) return PALU_ERR_INVALID_ARG;
  }
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const int d_h = h->d.head_dim;
  DecodeArgs a{};
  palu_cache c{};
  c.capacity = 1;
  fill_args(h, &c, batch, 0, a);
  a.rv = d_h;           // the merge's row: value-space outputs
  a.out_rv = 0;
  a.out = out;
  a.lse = lse;
  // split plan: like the decode kernels', in pages; partials of d_h floats must fit the workspace
  int cap = h->L.max_splits * h->ks.rv / d_h;
  if (cap > 256) cap = 256;
  if (cap < 1) return PALU_ERR_WORKSPACE;   // a handle whose partials cannot hold one d_h-wide split
  const int64_t units = (int64_t)batch * h->d.n_heads;
  int n_splits = 1, per = (int)(max_pages > 0 ? max_pages : 1);
  plan_splits(max_pages > 0 ? max_pages : 1, units, (int64_t)h->sm_count * paged_ctas_per_sm(pages->rank), cap, 8,
              &n_splits, &per);
  a.n_splits = n_splits;
  PagedArgs P{};
  P.pages = pages->pages;
  P.n_pages = pages->n_pages;
  P.capacity = pages->capacity;
  P.max_pages = (int)max_pages;
  P.dtype = to_dt(pages->dtype);
  P.rank = pages->rank;
  P.n_heads = h->d.n_heads;
  P.rope = h->d.mode == PALU_MODE_ROPE;
  P.q_pos = q_pos;
  P.rope_tab = a.rope;
  P.max_pos = a.max_pos;
  P.q = q;
  P.q_dtype = a.q_dtype;
  P.qscale = a.qscale;
  P.pages_per_split = per;
  P.err = a.err;
  P.wait_ns = a.wait_ns;
  P.m = a;
  cudaError_t e = launch_decode_paged(P, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return PALU_ERR_CUDA;
  if (!dense) return PALU_OK;
  return merge_dense_segment(h, a, dense, batch, d_h, q, q_pos, out, out_dense, lse, stream);
}

palu_status_t palu_debug_dequant(palu_attn_t h, const palu_cache* cache, int which, int batch, int64_t n_tokens,
                                 float* out, palu_stream_t stream) {
  if (!h || !out || (which != 0 && which != 1)) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  const palu_dtype_t dt = which == 0 ? h->d.k_dtype : h->d.v_dtype;
  if (dt != PALU_INT4) return PALU_ERR_INVALID_ARG;
  if (batch < 0 || batch > h->d.max_batch || n_tokens < 0 || n_tokens > cache->capacity) return PALU_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const cudaError_t e = launch_debug_dequant(which == 0 ? cache->hk : cache->hv,
                                             static_cast<const __half*>(which == 0 ? cache->k_scale : cache->v_scale),
                                             to_dt(dt), cache->capacity, h->n_g,
                                             which == 0 ? h->d.rank_k : h->d.rank_v, batch, n_tokens, out,
                                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

palu_status_t palu_debug_int4_operand(palu_attn_t h, const palu_cache* cache, int batch, int64_t n_tokens,
                                      uint16_t* codes, float* deq, palu_stream_t stream) {
  if (!h || !codes || (uintptr_t)codes % 2 || (uintptr_t)deq % 4) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  if (h->d.k_dtype != PALU_INT4) return PALU_ERR_INVALID_ARG;
  if (batch < 0 || batch > h->d.max_batch || n_tokens < 0 || n_tokens > cache->capacity) return PALU_ERR_INVALID_ARG;
  if (batch == 0 || n_tokens == 0) return PALU_OK;
  if (!tc_int4_debug_supported(h->n_g, h->d.rank_k, (int64_t)batch * cache->capacity)) return PALU_ERR_UNSUPPORTED;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const cudaError_t e = launch_debug_int4_operand(cache->hk, static_cast<const __half*>(cache->k_scale),
                                                  cache->capacity, h->n_g, batch, n_tokens, codes, deq,
                                                  reinterpret_cast<ErrWord*>(h->ws + h->L.err),
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

palu_status_t palu_debug_int4_dp2a(palu_attn_t h, const palu_cache* cache, int which, int batch, int64_t n_tokens,
                                   const int32_t* weights, int32_t* sums, palu_stream_t stream) {
  if (!h || (which != 0 && which != 1)) return PALU_ERR_INVALID_ARG;
  palu_status_t st = check_cache(h, cache);
  if (st != PALU_OK) return st;
  const palu_dtype_t dt = which == 0 ? h->d.k_dtype : h->d.v_dtype;
  const int rank = which == 0 ? h->d.rank_k : h->d.rank_v;
  if (dt != PALU_INT4) return PALU_ERR_INVALID_ARG;
  if (batch < 0 || batch > h->d.max_batch || n_tokens < 0 || n_tokens > cache->capacity) return PALU_ERR_INVALID_ARG;
  if (batch == 0 || n_tokens == 0) return PALU_OK;
  if (!weights || !sums || (uintptr_t)weights % 4 || (uintptr_t)sums % 4) return PALU_ERR_INVALID_ARG;
  if (rank != 256) return PALU_ERR_UNSUPPORTED;
  if (cudaSetDevice(h->device) != cudaSuccess) return PALU_ERR_CUDA;
  const cudaError_t e = launch_debug_int4_dp2a(which == 0 ? cache->hk : cache->hv, cache->capacity, h->n_g, batch,
                                               n_tokens, weights, sums, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

}  // extern "C"
