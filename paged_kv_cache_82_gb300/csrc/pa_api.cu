// pa_api.cu -- the C ABI of libpa: host-side validation, planning and
// launches.  Every entry point validates its arguments before launching
// anything and never synchronises the stream (pa_get_device_error excepted).
#include <math.h>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// One device-side error word per device (bits PA_DEV_ERR_*).
__device__ unsigned g_device_error;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  unsigned* err = nullptr;
  int num_sms = 0;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

// Address of the error word and the SM count of the current device.
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return nullptr;
    d.err = static_cast<unsigned*>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  return &d;
}

int elem_bytes(pa_dtype t) {
  switch (t) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
  }
  return 0;
}

bool valid_dtype(int t) { return t >= PA_F32 && t <= PA_NVFP4; }

// bytes of one (block, KV head) page of a cache of type t
int64_t page_bytes(pa_dtype t, int head_dim) {
  if (is_4bit(t)) return PA_PAGE_BYTES(t, head_dim);
  return (int64_t)PA_BLOCK_SIZE * head_dim * elem_bytes(t);
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// PA_OK, or why the cache geometry cannot be taken
pa_status cache_shape_status(int64_t num_blocks, int block_size,
                             int num_kv_heads, int head_dim) {
  if (num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  // row coordinates of the tensor maps are 32-bit
  if (num_blocks * (int64_t)num_kv_heads * PA_BLOCK_SIZE >= (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// the values last given to pa_set_wait_limit_ns / pa_test_skip_copy (both
// are written together into every pipelined translation unit)
std::mutex g_hooks_mutex;
uint64_t g_hook_wait_ns = kWaitLimitNs;
long long g_hook_skip = -1;

thread_local ProfileEvents t_profile;
thread_local uint64_t t_launches = 0;

}  // namespace

ProfileEvents& profile_events() { return t_profile; }

void count_launch() { ++t_launches; }

bool encode_cache_tensor_maps(const AttnArgs& a, CUtensorMap* tk,
                              CUtensorMap* tv, int box_rows) {
  // 4-bit pages go by untiled bulk copies: no tensor map
  if (is_4bit(a.cache_dtype)) return true;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int eb = elem_bytes(a.cache_dtype);
  const cuuint64_t rows =
      (cuuint64_t)a.num_blocks * a.num_kv_heads * PA_BLOCK_SIZE;
  const cuuint64_t row_bytes = (cuuint64_t)a.head_dim * eb;
  // Pages are viewed as rows of 128-byte segments: [rows][row_bytes/128][128 B]
  // so that one box = one (block, head) page with the 128-byte swizzle.
  const cuuint32_t inner = 128 / eb;
  const cuuint32_t segs = (cuuint32_t)(row_bytes / 128);
  CUtensorMapDataType dt =
      eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const void* ptrs[2] = {a.k_cache, a.v_cache};
  CUtensorMap* maps[2] = {tk, tv};
  for (int k = 0; k < 2; ++k) {
    CUresult res;
    if (segs == 1) {
      cuuint64_t dims[2] = {inner, rows};
      cuuint64_t strides[1] = {row_bytes};
      cuuint32_t box[2] = {inner, (cuuint32_t)box_rows};
      cuuint32_t es[2] = {1, 1};
      res = fn(maps[k], dt, 2, const_cast<void*>(ptrs[k]), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      cuuint64_t dims[3] = {inner, segs, rows};
      cuuint64_t strides[2] = {128, row_bytes};
      cuuint32_t box[3] = {inner, segs, (cuuint32_t)box_rows};
      cuuint32_t es[3] = {1, 1, 1};
      res = fn(maps[k], dt, 3, const_cast<void*>(ptrs[k]), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (res != CUDA_SUCCESS) return false;
  }
  return true;
}

bool encode_prefill_tensor_maps(const AttnArgs& a, TcMaps* m) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || a.head_dim != 128) return false;
  const int G = a.num_q_heads / a.num_kv_heads;
  const cuuint32_t tp = (cuuint32_t)(128 / G);
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const cuuint32_t es[3] = {1, 1, 1};
  // q [token][head][128]: a box is 64 columns of G heads of 128/G tokens
  {
    cuuint64_t dims[3] = {128, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_tokens};
    cuuint64_t strides[2] = {256, (cuuint64_t)a.num_q_heads * 256};
    cuuint32_t box[3] = {64, (cuuint32_t)G, tp};
    if (fn(&m->q, dt, 3, const_cast<void*>(a.q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  // caches [row][128]: a box is 64 columns of one 16-row page; FP8 caches
  // [row][128 bytes]: a box is one whole page (widened in shared memory)
  const cuuint64_t rows = (cuuint64_t)a.num_blocks * a.num_kv_heads * PA_BLOCK_SIZE;
  const void* ptrs[2] = {a.k_cache, a.v_cache};
  CUtensorMap* maps[2] = {&m->k, &m->v};
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
  for (int k = 0; k < 2; ++k) {
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {fp8 ? 128u : 256u};
    cuuint32_t box[2] = {fp8 ? 128u : 64u, PA_BLOCK_SIZE};
    if (fn(maps[k], fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : dt, 2,
           const_cast<void*>(ptrs[k]), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
  }
  return "PA_ERR_UNKNOWN";
}

pa_status pa_reshape_and_cache(const void* key, const void* value,
                               pa_dtype kv_dtype, int64_t num_tokens,
                               int64_t key_stride, int64_t value_stride,
                               void* k_cache, void* v_cache,
                               pa_dtype cache_dtype, int64_t num_blocks,
                               int block_size, int num_kv_heads, int head_dim,
                               const int64_t* slot_mapping, float k_scale,
                               float v_scale, pa_stream_t stream) {
  if (!valid_dtype(kv_dtype) || !valid_dtype(cache_dtype))
    return PA_ERR_INVALID_ARG;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (pa_status st = cache_shape_status(num_blocks, block_size, num_kv_heads,
                                        head_dim))
    return st;
  if (kv_dtype == PA_FP8_E4M3 || is_4bit(kv_dtype)) return PA_ERR_UNSUPPORTED;
  if (cache_dtype != kv_dtype && cache_dtype != PA_FP8_E4M3 &&
      !is_4bit(cache_dtype))
    return PA_ERR_UNSUPPORTED;
  if ((cache_dtype == PA_FP8_E4M3 || cache_dtype == PA_NVFP4) &&
      !(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0 && v_scale > 0))
    return PA_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (key_stride < row || value_stride < row) return PA_ERR_INVALID_ARG;
  if (!k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
  const int ib = elem_bytes(kv_dtype);
  const int cb = is_4bit(cache_dtype) ? 16 : elem_bytes(cache_dtype);
  if (!aligned(key, ib) || !aligned(value, ib) || !aligned(k_cache, cb) ||
      !aligned(v_cache, cb) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  const size_t cache_bytes =
      (size_t)num_blocks * num_kv_heads * page_bytes(cache_dtype, head_dim);
  const size_t in_bytes_k = ((size_t)(num_tokens - 1) * key_stride + row) * ib;
  const size_t in_bytes_v = ((size_t)(num_tokens - 1) * value_stride + row) * ib;
  if (overlaps(k_cache, cache_bytes, v_cache, cache_bytes) ||
      overlaps(key, in_bytes_k, k_cache, cache_bytes) ||
      overlaps(key, in_bytes_k, v_cache, cache_bytes) ||
      overlaps(value, in_bytes_v, k_cache, cache_bytes) ||
      overlaps(value, in_bytes_v, v_cache, cache_bytes))
    return PA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return PA_ERR_CUDA;
  if (is_4bit(cache_dtype)) {
    cudaError_t e4 = launch_reshape_4bit(
        key, value, kv_dtype, num_tokens, key_stride, value_stride, k_cache,
        v_cache, cache_dtype, num_blocks, num_kv_heads, head_dim, slot_mapping,
        k_scale, v_scale, di->err, reinterpret_cast<cudaStream_t>(stream));
    return e4 == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  // 8-element vectors: 16 bytes (16-bit) or 32 bytes (fp32) on the input
  // side, 8 / 16 / 32 bytes on the cache side
  const size_t va = 8 * (size_t)ib;
  const bool vector_ok = aligned(key, va) && aligned(value, va) &&
                         (key_stride * ib) % va == 0 &&
                         (value_stride * ib) % va == 0 &&
                         aligned(k_cache, 8 * (size_t)cb) &&
                         aligned(v_cache, 8 * (size_t)cb);
  cudaError_t e = launch_reshape_and_cache(
      key, value, kv_dtype, num_tokens, key_stride, value_stride, k_cache,
      v_cache, cache_dtype, num_blocks, num_kv_heads, head_dim, slot_mapping,
      k_scale, v_scale, vector_ok, di->err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_dtype cache_dtype,
                         int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, const int64_t* block_mapping,
                         int64_t num_pairs, pa_stream_t stream) {
  if (!valid_dtype(cache_dtype)) return PA_ERR_INVALID_ARG;
  if (pa_status st = cache_shape_status(num_blocks, block_size, num_kv_heads,
                                        head_dim))
    return st;
  if (num_pairs < 0 || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_mapping || !aligned(block_mapping, 8)) return PA_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
  const int64_t block_bytes =
      (int64_t)num_kv_heads * page_bytes(cache_dtype, head_dim);
  if (overlaps(k_cache, (size_t)(num_blocks * block_bytes), v_cache,
               (size_t)(num_blocks * block_bytes)))
    return PA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return PA_ERR_CUDA;
  cudaError_t e = launch_copy_blocks(k_cache, v_cache, num_blocks, block_bytes,
                                     block_mapping, num_pairs, di->err,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

pa_status workspace_size_impl(int64_t num_tokens, int num_q_heads,
                              int num_kv_heads, int head_dim, int num_seqs,
                              int max_query_len, int max_seq_len, int window,
                              bool cascade, size_t* bytes) {
  if (!bytes) return PA_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || max_query_len < 0 || max_seq_len < 0 ||
      window < 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  const DeviceInfo* di = device_info();
  if (!di) return PA_ERR_CUDA;
  const AttnPlan pl = make_plan(num_tokens, num_q_heads, num_kv_heads, head_dim,
                                num_seqs, max_query_len, max_seq_len,
                                di->num_sms, window, cascade);
  *bytes = pl.total_bytes;
  return PA_OK;
}

pa_status attention_impl(const void* q, pa_dtype q_dtype, const void* k_cache,
                         const void* v_cache, pa_dtype cache_dtype,
                         int64_t num_blocks, int block_size, int num_q_heads,
                         int num_kv_heads, int head_dim,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens,
                         const int32_t* query_start_loc, int num_seqs,
                         int64_t num_tokens, int max_query_len, int max_seq_len,
                         float scale, float k_scale, float v_scale, int window,
                         int cascade_blocks, void* out, void* workspace,
                         size_t workspace_bytes, pa_stream_t stream) {
  if (window < 0 || cascade_blocks < 0) return PA_ERR_INVALID_ARG;
  if (!valid_dtype(q_dtype) || !valid_dtype(cache_dtype))
    return PA_ERR_INVALID_ARG;
  if (pa_status st = cache_shape_status(num_blocks, block_size, num_kv_heads,
                                        head_dim))
    return st;
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (q_dtype == PA_FP8_E4M3 || is_4bit(q_dtype)) return PA_ERR_UNSUPPORTED;
  const bool quantised = cache_dtype == PA_FP8_E4M3 || is_4bit(cache_dtype);
  if (!quantised && cache_dtype != q_dtype) return PA_ERR_UNSUPPORTED;
  if (quantised && q_dtype == PA_F32) return PA_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if ((cache_dtype == PA_FP8_E4M3 || cache_dtype == PA_NVFP4) &&
      !(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0 && v_scale > 0))
    return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || max_seq_len < 0 ||
      max_blocks_per_seq < 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PA_OK;
  if ((int64_t)max_blocks_per_seq * PA_BLOCK_SIZE < max_seq_len ||
      cascade_blocks > max_blocks_per_seq)
    return PA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens ||
      !query_start_loc || !out)
    return PA_ERR_INVALID_ARG;
  const int qb = elem_bytes(q_dtype);
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 128) ||
      !aligned(v_cache, 128) || !aligned(block_tables, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return PA_ERR_INVALID_ARG;
  const size_t qo_bytes = (size_t)num_tokens * num_q_heads * head_dim * qb;
  const size_t cache_bytes =
      (size_t)num_blocks * num_kv_heads * page_bytes(cache_dtype, head_dim);
  const DeviceInfo* di = device_info();
  if (!di) return PA_ERR_CUDA;
  AttnPlan plan = make_plan(num_tokens, num_q_heads, num_kv_heads, head_dim,
                            num_seqs, max_query_len, max_seq_len, di->num_sms,
                            window);
  AttnArgs a{};
  a.q = q;
  a.q_dtype = q_dtype;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache_dtype = cache_dtype;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.scale = scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out = out;
  a.workspace = workspace;
  a.err = di->err;
  a.window = plan.window;
  // a shared prefix runs as a cascade where the step's types and shapes
  // allow it; elsewhere the hint is not used (the same attention, computed
  // over every request's whole row)
  a.cascade_blocks = cascade_blocks;
  if (cascade_blocks > 0 && cascade_supported(a))
    plan = make_plan(num_tokens, num_q_heads, num_kv_heads, head_dim, num_seqs,
                     max_query_len, max_seq_len, di->num_sms, window, true);
  else
    a.cascade_blocks = 0;
  const bool fast = fast_path_supported(a);
  if (fast) {
    if (workspace_bytes < plan.total_bytes) return PA_ERR_INVALID_ARG;
    if (plan.total_bytes > 0 && (!workspace || !aligned(workspace, 256)))
      return PA_ERR_INVALID_ARG;
  }
  if (overlaps(out, qo_bytes, q, qo_bytes) ||
      overlaps(out, qo_bytes, k_cache, cache_bytes) ||
      overlaps(out, qo_bytes, v_cache, cache_bytes) ||
      (fast && overlaps(out, qo_bytes, workspace, plan.total_bytes)))
    return PA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (fast && plan.window > 0) {
    // the kernels of the step see each request through the window: its
    // blocks from the one holding its first visible key (workspace)
    e = launch_window_view(a, plan, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.block_tables = reinterpret_cast<const int32_t*>(ws + plan.off_win_bt);
    a.seq_lens = reinterpret_cast<const int32_t*>(ws + plan.off_win_sl);
    a.max_blocks_per_seq = plan.win_blocks;
    a.max_seq_len = plan.win_max_seq_len;
  }
  if (fast) {
    // prefill tiles go to the tensor-core kernel where it takes the step's
    // types (else the attention kernel runs them on the warp-level MMA)
    TcMaps tc;
    const bool use_tc = (plan.has_prefill || plan.cascade) && tc_prefill_supported(a) &&
                        encode_prefill_tensor_maps(a, &tc);
    CUtensorMap tk{}, tv{};
    if (!encode_cache_tensor_maps(a, &tk, &tv, decode_box_rows(a, use_tc)))
      return PA_ERR_CUDA;
    e = launch_attention_fast(a, plan, tk, tv, use_tc ? &tc : nullptr,
                              di->num_sms, s);
  } else {
    e = launch_attention_generic(a, s);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status pa_attention_workspace_size(int64_t num_tokens, int num_q_heads,
                                      int num_kv_heads, int head_dim,
                                      int num_seqs, int max_query_len,
                                      int max_seq_len, size_t* bytes) {
  return workspace_size_impl(num_tokens, num_q_heads, num_kv_heads, head_dim,
                             num_seqs, max_query_len, max_seq_len, 0, false, bytes);
}

pa_status pa_attention_cascade_workspace_size(int64_t num_tokens, int num_q_heads,
                                              int num_kv_heads, int head_dim,
                                              int num_seqs, int max_query_len,
                                              int max_seq_len, size_t* bytes) {
  return workspace_size_impl(num_tokens, num_q_heads, num_kv_heads, head_dim,
                             num_seqs, max_query_len, max_seq_len, 0, true, bytes);
}

pa_status pa_attention_window_workspace_size(int64_t num_tokens,
                                             int num_q_heads, int num_kv_heads,
                                             int head_dim, int num_seqs,
                                             int max_query_len, int max_seq_len,
                                             int sliding_window, size_t* bytes) {
  return workspace_size_impl(num_tokens, num_q_heads, num_kv_heads, head_dim,
                             num_seqs, max_query_len, max_seq_len,
                             sliding_window, false, bytes);
}

pa_status pa_attention(const void* q, pa_dtype q_dtype, const void* k_cache,
                       const void* v_cache, pa_dtype cache_dtype,
                       int64_t num_blocks, int block_size, int num_q_heads,
                       int num_kv_heads, int head_dim,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens,
                       const int32_t* query_start_loc, int num_seqs,
                       int64_t num_tokens, int max_query_len, int max_seq_len,
                       float scale, float k_scale, float v_scale, void* out,
                       void* workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  return attention_impl(q, q_dtype, k_cache, v_cache, cache_dtype, num_blocks,
                        block_size, num_q_heads, num_kv_heads, head_dim,
                        block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_tokens, max_query_len,
                        max_seq_len, scale, k_scale, v_scale, 0, 0, out, workspace,
                        workspace_bytes, stream);
}

pa_status pa_attention_cascade(const void* q, pa_dtype q_dtype, const void* k_cache,
                               const void* v_cache, pa_dtype cache_dtype,
                               int64_t num_blocks, int block_size, int num_q_heads,
                               int num_kv_heads, int head_dim,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens,
                               const int32_t* query_start_loc, int num_seqs,
                               int64_t num_tokens, int max_query_len,
                               int max_seq_len, float scale, float k_scale,
                               float v_scale, int common_prefix_blocks, void* out,
                               void* workspace, size_t workspace_bytes,
                               pa_stream_t stream) {
  return attention_impl(q, q_dtype, k_cache, v_cache, cache_dtype, num_blocks,
                        block_size, num_q_heads, num_kv_heads, head_dim,
                        block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_tokens, max_query_len,
                        max_seq_len, scale, k_scale, v_scale, 0, common_prefix_blocks,
                        out, workspace, workspace_bytes, stream);
}

pa_status pa_attention_window(const void* q, pa_dtype q_dtype,
                              const void* k_cache, const void* v_cache,
                              pa_dtype cache_dtype, int64_t num_blocks,
                              int block_size, int num_q_heads, int num_kv_heads,
                              int head_dim, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int num_seqs,
                              int64_t num_tokens, int max_query_len,
                              int max_seq_len, float scale, float k_scale,
                              float v_scale, int sliding_window, void* out,
                              void* workspace, size_t workspace_bytes,
                              pa_stream_t stream) {
  return attention_impl(q, q_dtype, k_cache, v_cache, cache_dtype, num_blocks,
                        block_size, num_q_heads, num_kv_heads, head_dim,
                        block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_tokens, max_query_len,
                        max_seq_len, scale, k_scale, v_scale, sliding_window, 0,
                        out, workspace, workspace_bytes, stream);
}

pa_status pa_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) ns = kWaitLimitNs;
  if (ns < 100000ull || ns > 60000000000ull) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_hooks_mutex);
  if (set_pipeline_hooks_fast(ns, g_hook_skip) != cudaSuccess ||
      set_pipeline_hooks_tc(ns, g_hook_skip) != cudaSuccess)
    return PA_ERR_CUDA;
  g_hook_wait_ns = ns;
  return PA_OK;
}

pa_status pa_test_skip_copy(int64_t stage) {
  if (stage < -1) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_hooks_mutex);
  if (set_pipeline_hooks_fast(g_hook_wait_ns, stage) != cudaSuccess ||
      set_pipeline_hooks_tc(g_hook_wait_ns, stage) != cudaSuccess)
    return PA_ERR_CUDA;
  g_hook_skip = stage;
  return PA_OK;
}

pa_status pa_set_debug_bounds(int enable) {
  return enable ? PA_OK : PA_ERR_UNSUPPORTED;
}

pa_status pa_launch_count(uint64_t* count) {
  if (!count) return PA_ERR_INVALID_ARG;
  *count = t_launches;
  return PA_OK;
}

pa_status pa_set_profile_events(pa_event_t start, pa_event_t stop) {
  if ((start == nullptr) != (stop == nullptr)) return PA_ERR_INVALID_ARG;
  profile_events().start = reinterpret_cast<cudaEvent_t>(start);
  profile_events().stop = reinterpret_cast<cudaEvent_t>(stop);
  return PA_OK;
}

pa_status pa_get_device_error(pa_stream_t stream, uint32_t* flags) {
  if (!flags) return PA_ERR_INVALID_ARG;
  *flags = 0;
  const DeviceInfo* di = device_info();
  if (!di) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess)
    return PA_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
    return PA_ERR_CUDA;
  *flags = v;
  return v ? PA_ERR_DEVICE : PA_OK;
}

}  // extern "C"
