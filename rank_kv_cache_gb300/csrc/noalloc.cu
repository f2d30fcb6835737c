// Decode entry point for callers that cannot allocate device memory.
//
// Some callers run where cudaMalloc is not available to them: a plugin whose host
// process owns every allocation, an inference engine with a fixed memory plan, or
// code that must not allocate once serving has started. For them,
// palu_decode_attn_noalloc runs the absorbed-mode decode (query absorption,
// split-T attention, split merge) with its scratch in the fixed device array
// below instead of a caller-provided workspace. It calls no allocating routine.
#include <mutex>

#include "palu_attn.h"
#include "internal.h"

using namespace palu;

namespace {

// Fixed scratch: error word, absorbed queries and split partials. Every GPU that
// loads this library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
char* g_scratch[kMaxDevices];  // device address of g_noalloc_scratch, per device
int g_sms[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Once per device, with that device current: look up the array's device address.
palu_status_t scratch_for(int dev, char** ptr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return PALU_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PALU_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PALU_ERR_CUDA;
    g_scratch[dev] = static_cast<char*>(p);
    g_sms[dev] = n;
  }
  *ptr = g_scratch[dev];
  *sms = g_sms[dev];
  return PALU_OK;
}

}  // namespace

extern "C" palu_status_t palu_decode_attn_noalloc(const palu_attn_desc* desc, const void* B_k, const void* q,
                                                  const palu_cache* cache, const int32_t* seq_lens, int batch,
                                                  int64_t max_seq_len, float* out, float* lse,
                                                  palu_stream_t stream) {
  size_t ws_unused = 0;
  palu_status_t st = palu_attn_workspace_size(desc, &ws_unused);  // validates the descriptor
  if (st != PALU_OK) return st;
  if (desc->mode != PALU_MODE_ABSORBED) return PALU_ERR_UNSUPPORTED;
  if (desc->group_size > 8) return PALU_ERR_UNSUPPORTED;   // the CUDA-core kernel takes up to 8 heads a group
  if (desc->flags & PALU_FLAG_ALIBI) return PALU_ERR_UNSUPPORTED;   // this entry point takes no positions
  if (batch < 0 || batch > desc->max_batch) return PALU_ERR_INVALID_ARG;
  if (batch == 0) return PALU_OK;
  if (!B_k || (uintptr_t)B_k % 16 || !q || (uintptr_t)q % 4 || !seq_lens || !out || (uintptr_t)out % 16)
    return PALU_ERR_INVALID_ARG;
  if (!cache || !cache->hk || !cache->hv || cache->capacity <= 0) return PALU_ERR_INVALID_ARG;
  if ((uintptr_t)cache->hk % 16 || (uintptr_t)cache->hv % 16) return PALU_ERR_INVALID_ARG;
  if (desc->k_dtype == PALU_INT4 && (!cache->k_scale || (uintptr_t)cache->k_scale % 2)) return PALU_ERR_INVALID_ARG;
  if (desc->v_dtype == PALU_INT4 && (!cache->v_scale || (uintptr_t)cache->v_scale % 2)) return PALU_ERR_INVALID_ARG;
  if (max_seq_len < 0 || max_seq_len > desc->max_tokens || max_seq_len > cache->capacity)
    return PALU_ERR_INVALID_ARG;

  const int n_g = desc->n_heads / desc->group_size;
  const size_t bh = (size_t)batch * desc->n_heads;
  const size_t fixed = 256 + align256(bh * desc->rank_k * sizeof(float));
  const size_t per_split = bh * desc->rank_v * sizeof(float) + bh * sizeof(float2);
  if (fixed + per_split + 512 > kNoAllocScratchBytes) return PALU_ERR_WORKSPACE;  // beyond the fixed scratch

  // the scratch address is per device: the stream must belong to the current device
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, stream_dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PALU_ERR_CUDA;
  if (cudaStreamGetDevice(s, &stream_dev) != cudaSuccess) {
    cudaGetLastError();
    return PALU_ERR_INVALID_ARG;
  }
  if (stream_dev != dev) return PALU_ERR_INVALID_ARG;
  char* scratch = nullptr;
  int sms = 0;
  st = scratch_for(dev, &scratch, &sms);
  if (st != PALU_OK) return st;

  // split-T plan as in palu_decode_attn, capped by the fixed scratch
  const int64_t tiles = max_seq_len > 0 ? (max_seq_len + kSimtTile - 1) / kSimtTile : 1;
  const int64_t units = (int64_t)batch * n_g;
  int64_t splits = (2LL * sms + units - 1) / units;
  const int64_t fit = (int64_t)((kNoAllocScratchBytes - fixed - 512) / per_split);
  int64_t cap = tiles < 256 ? tiles : 256;
  if (cap > fit) cap = fit;
  if (splits > cap) splits = cap;
  if (splits < 1) splits = 1;
  const int64_t tps = (tiles + splits - 1) / splits;
  splits = (tiles + tps - 1) / tps;

  DecodeArgs a{};
  a.hk = cache->hk;
  a.hv = cache->hv;
  a.k_scale = static_cast<const __half*>(cache->k_scale);
  a.v_scale = static_cast<const __half*>(cache->v_scale);
  a.capacity = cache->capacity;
  a.n_heads = desc->n_heads;
  a.n_g = n_g;
  a.s = desc->group_size;
  a.dh = desc->head_dim;
  a.rk = desc->rank_k;
  a.rv = desc->rank_v;
  a.k_dtype = (int)desc->k_dtype;
  a.v_dtype = (int)desc->v_dtype;
  a.bk_dtype = (int)desc->bk_dtype;
  a.seq_lens = seq_lens;
  a.positions = nullptr;
  a.batch = batch;
  a.max_seq_len = (int)max_seq_len;
  a.max_pos = 1;
  a.bk = B_k;
  a.bkt = nullptr;
  a.rope = nullptr;
  a.err = reinterpret_cast<ErrWord*>(scratch);
  float* qbuf = reinterpret_cast<float*>(scratch + 256);
  a.qbuf = qbuf;
  a.part_o = reinterpret_cast<float*>(scratch + fixed);
  a.part_ml = reinterpret_cast<float2*>(scratch + fixed + align256((size_t)splits * bh * desc->rank_v * sizeof(float)));
  a.n_splits = (int)splits;
  a.tiles_per_split = (int)tps;

  const float qscale = float(1.4426950408889634 / sqrt((double)desc->head_dim));
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, s);  // the error word starts at zero on every call
  if (e == cudaSuccess) e = launch_qprep(kAbsorbed, q, (int)desc->q_dtype, a, nullptr, qscale, qbuf, s);
  if (e == cudaSuccess) e = launch_decode_simt(kAbsorbed, a, s);
  if (e == cudaSuccess) e = launch_combine(a, out, lse, s);
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}
