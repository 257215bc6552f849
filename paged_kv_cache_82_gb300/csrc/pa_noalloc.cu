// pa_noalloc.cu -- pa_attention for callers that cannot allocate device
// memory.
//
// pa_attention needs a caller-provided workspace of a size only known per
// step.  Some callers have no way to obtain one: a serving engine that hands
// all free HBM to its KV-cache pool at start-up and allocates nothing after,
// or code that must not call cudaMalloc / cudaFree because those may
// synchronise the device in the middle of a step.  For them this file keeps
// one fixed scratch buffer in device memory, declared as a file-scope
// __device__ array, and runs the same attention with it.
//
// The array is part of the library image: every GPU that loads the library
// holds it (PA_NOALLOC_SCRATCH_BYTES) until the process exits.  Host code
// cannot use the array's name as a device address; its address is looked up
// once per device with cudaGetSymbolAddress, on the first call made while
// that device is current, and kept for the life of the process (a
// cudaDeviceReset invalidates it, as it does every other device address the
// library holds; pa.h says so).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// The workspace of every decode step holds the split-K partial slots of all
// resident attention CTAs, whatever the batch: kPartialBytesPerSm per SM.
// The scratch must hold that floor on the largest GPU this library targets
// (160 SMs; GB300 enables 152) with room to spare for the step's lists,
// otherwise every decode call would be rejected.  A build with more resident
// CTAs per SM (PA_CTAS_PER_SM) that breaks this must raise the size.
constexpr size_t kMaxTargetSms = 160;
static_assert(pa::kPartialBytesPerSm * kMaxTargetSms + (2u << 20) <=
                  (size_t)PA_NOALLOC_SCRATCH_BYTES,
              "PA_NOALLOC_SCRATCH_BYTES is below the decode workspace floor");

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up on the
// first call for that device), or nullptr on failure.
void* scratch_address(pa_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *st = PA_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = PA_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *st = PA_ERR_CUDA;
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  *st = PA_OK;
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" pa_status pa_attention_noalloc(
    const void* q, pa_dtype q_dtype, const void* k_cache, const void* v_cache,
    pa_dtype cache_dtype, int64_t num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* seq_lens,
    const int32_t* query_start_loc, int num_seqs, int64_t num_tokens,
    int max_query_len, int max_seq_len, float scale, float k_scale,
    float v_scale, void* out, pa_stream_t stream) {
  // the scratch the step needs must fit in the fixed array
  size_t need = 0;
  pa_status st = pa_attention_workspace_size(num_tokens, num_q_heads,
                                             num_kv_heads, head_dim, num_seqs,
                                             max_query_len, max_seq_len, &need);
  if (st != PA_OK) return st;
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_INVALID_ARG;
  void* scratch = scratch_address(&st);
  if (scratch == nullptr) return st;
  // Nothing in the scratch has to start at zero: every byte the attention
  // reads is written earlier in the same call.
  return pa_attention(q, q_dtype, k_cache, v_cache, cache_dtype, num_blocks,
                      block_size, num_q_heads, num_kv_heads, head_dim,
                      block_tables, max_blocks_per_seq, seq_lens,
                      query_start_loc, num_seqs, num_tokens, max_query_len,
                      max_seq_len, scale, k_scale, v_scale, out, scratch,
                      (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
