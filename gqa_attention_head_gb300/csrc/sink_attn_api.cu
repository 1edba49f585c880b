// sink_attn_api.cu — the extern "C" boundary declared in include/sink_attn.h:
// argument validation, TMA tensor-map encoding, workspace layout, device error word,
// and the launches. Nothing here allocates device memory or synchronises, except
// sink_attn_read_device_error, whose documented purpose is to synchronise.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "sink_attn.h"

namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s per pipeline wait
constexpr int kMaxDevices = 64;

// Test switch of the decode launches (sink_attn_debug_decode_withhold_page): the first
// page of (chunk 0, kv head 0, sequence 0) withheld, and the pipeline-wait limit.
std::atomic<int> g_decode_withhold{0};
std::atomic<uint64_t> g_decode_wait_ns{kWaitTimeoutNs};

// Device error word: set by kernels (atomicOr of SINK_ATTN_DEVERR_* bits),
// read and cleared by sink_attn_read_device_error.
__device__ unsigned g_device_error;

std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool current_device(int& dev) {
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return dev >= 0 && dev < kMaxDevices;
}

// Device address of g_device_error on the current device (looked up once per device).
unsigned* device_error_word() {
  int dev;
  if (!current_device(dev)) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

int num_sms_current() {
  int dev;
  if (!current_device(dev)) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// bf16 [rows][heads][dim] as a 3-D map {dim, heads, rows}, box {64, box_heads, box_rows},
// 128-byte swizzle (each box row is exactly 128 bytes; a box lands as box_rows x box_heads
// rows of 128 bytes, heads fastest).
bool encode_3d(CUtensorMap* m, const void* base, uint64_t dim, uint64_t heads, uint64_t rows,
               uint32_t box_rows, uint32_t box_heads = 1) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[3] = {dim, heads, rows};
  cuuint64_t gstride[2] = {dim * 2, heads * dim * 2};
  cuuint32_t box[3] = {64, box_heads, box_rows};
  cuuint32_t estride[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][dim] as a 2-D map {dim, rows}, box {64, box_rows}, 128-byte swizzle.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t dim, uint64_t rows, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {dim, rows};
  cuuint64_t gstride[1] = {dim * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 codes [rows][dim] (dim 64 or 128 bytes) as a 2-D uint8 map {dim, rows}, box
// {dim, box_rows}: one box holds whole rows, swizzled at the row's width (64 or 128 bytes).
bool encode_2d_u8(CUtensorMap* m, const void* base, uint64_t dim, uint64_t rows,
                  uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {dim, rows};
  cuuint64_t gstride[1] = {dim};
  cuuint32_t box[2] = {(cuuint32_t)dim, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             dim == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout for `cmax` chunks: o_part [B][Hq][cmax][D] fp32, then lse_part
// [B][Hq][cmax] fp32 at a 256-byte boundary. Zero when no sequence needs two chunks.
// Scratch of sink_attn_prefill_from_host: per range at most 2 (S + 1) int32 offsets, then
// the sinks (fp32).
size_t from_host_scratch_bytes(int64_t num_seqs, int64_t hq, int64_t n_ranges) {
  return (size_t)(n_ranges * 2 * (num_seqs + 1) + hq) * 4;
}

size_t workspace_bytes_for(int64_t batch, int64_t hq, int64_t d, int64_t cmax) {
  if (cmax <= 1) return 0;
  return align_up((size_t)(batch * hq * cmax * d) * 4, 256) + (size_t)(batch * hq * cmax) * 4;
}

}  // namespace

extern "C" {

const char* sink_attn_status_string(sink_attn_status s) {
  switch (s) {
    case SINK_ATTN_OK: return "ok";
    case SINK_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case SINK_ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case SINK_ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case SINK_ATTN_ERR_CUDA: return "CUDA error";
    case SINK_ATTN_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

void sink_attn_debug_decode_withhold_page(int32_t enable, uint64_t wait_limit_ns) {
  g_decode_wait_ns.store(enable ? wait_limit_ns : kWaitTimeoutNs);
  g_decode_withhold.store(enable ? 1 : 0);
}

int32_t sink_attn_num_sms(void) { return num_sms_current(); }

size_t sink_attn_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                        int32_t max_seq_len, int32_t kv_chunk) {
  if (batch <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0 || kv_chunk <= 0)
    return 0;
  return workspace_bytes_for(batch, num_q_heads, head_dim,
                             sa::decode_max_chunks(max_seq_len, 0, kv_chunk));
}

}  // extern "C"

namespace {

sink_attn_status prefill_impl(const sink_attn_bf16* q, const sink_attn_bf16* k,
                              const sink_attn_bf16* v, const float* sinks,
                              const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                              int32_t max_seqlen, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t window, float scale, sink_attn_bf16* out,
                              float* lse, sink_attn_stream_t stream,
                              const int32_t* cu_seqlens_k = nullptr, int32_t total_k = 0,
                              int32_t max_seqlen_k = 0) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return SINK_ATTN_ERR_INVALID_ARG;
  const bool kv_own = cu_seqlens_k != nullptr;
  if (kv_own && (total_k < 0 || max_seqlen_k < max_seqlen || !aligned4(cu_seqlens_k)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return SINK_ATTN_OK;
  if (!q || !k || !v || !out || !cu_seqlens) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned4(cu_seqlens) || (sinks && !aligned4(sinks)) || (lse && !aligned4(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if ((int64_t)total_tokens * num_q_heads >= ((int64_t)1 << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  const int32_t rows_k = kv_own ? total_k : total_tokens;
  if (rows_k == 0) return SINK_ATTN_ERR_INVALID_ARG;  // queries need their keys
  const int64_t n_qt = (max_seqlen + 127) / 128;
  if (n_qt * num_seqs * num_q_heads >= ((int64_t)1 << 31)) return SINK_ATTN_ERR_UNSUPPORTED;

  sa::PrefillLaunch a{};
  a.err = device_error_word();
  a.num_sms = num_sms_current();
  if (!a.err || a.num_sms <= 0) return SINK_ATTN_ERR_CUDA;
  a.band = (!kv_own && sa::prefill_band_applies(head_dim, window, num_q_heads, num_kv_heads,
                                                total_tokens, num_seqs, a.num_sms))
               ? 1
               : 0;
  const bool maps_ok =
      a.band ? encode_3d(&a.tm_q, q, head_dim, num_q_heads, total_tokens, 16, 8) &&
                   encode_3d(&a.tm_o, out, head_dim, num_q_heads, total_tokens, 4, 8) &&
                   encode_3d(&a.tm_k, k, head_dim, num_kv_heads, rows_k, 160) &&
                   encode_3d(&a.tm_v, v, head_dim, num_kv_heads, rows_k, 160)
             : encode_3d(&a.tm_q, q, head_dim, num_q_heads, total_tokens, 128) &&
                   encode_3d(&a.tm_k, k, head_dim, num_kv_heads, rows_k, 128) &&
                   encode_3d(&a.tm_v, v, head_dim, num_kv_heads, rows_k, 128);
  if (!maps_ok) return SINK_ATTN_ERR_CUDA;
  a.cu_seqlens = cu_seqlens;
  a.kv_lens = nullptr;
  a.page_table = nullptr;
  a.max_pages = a.num_pages = 0;
  a.max_kv = kv_own ? max_seqlen_k : 0;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_k = rows_k;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.num_seqs = num_seqs;
  a.total_tokens = total_tokens;
  a.max_seqlen = max_seqlen;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.window = window;
  a.scale = scale;
  a.timeout_ns = kWaitTimeoutNs;
  return sa::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

// k_cache/v_cache: bf16 pages, or (k_scale non-null) e4m3 code pages with row scales.
sink_attn_status decode_impl(const sink_attn_bf16* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, int32_t num_pages,
                             int32_t page_size,
                             const int32_t* page_table, int32_t max_pages_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             const float* sinks, int32_t window, float scale, int32_t kv_chunk,
                             void* workspace, size_t workspace_bytes, sink_attn_bf16* out,
                             float* lse, sink_attn_stream_t stream) {
  const bool fp8 = k_scale != nullptr || v_scale != nullptr;
  if (batch < 0 || max_seq_len < 0 || num_pages < 0 || max_pages_per_seq < 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (page_size != 16) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > 16) return SINK_ATTN_ERR_UNSUPPORTED;
  if (kv_chunk <= 0 || kv_chunk % page_size != 0) return SINK_ATTN_ERR_INVALID_ARG;
  if (batch == 0) return SINK_ATTN_OK;
  if (batch > 65535 || num_kv_heads > 65535) return SINK_ATTN_ERR_UNSUPPORTED;
  if (!q || !out || !seq_lens) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned4(seq_lens) || (sinks && !aligned4(sinks)) ||
      (lse && !aligned4(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  // With no cache positions at all every output is zero; the kernel still runs to
  // write them, reading no page. Otherwise the cache and page table must exist.
  const bool has_cache = max_seq_len > 0;
  if (has_cache) {
    if (num_pages <= 0 || !k_cache || !v_cache || !page_table || max_pages_per_seq <= 0)
      return SINK_ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned4(page_table))
      return SINK_ATTN_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
      return SINK_ATTN_ERR_INVALID_ARG;
    if ((int64_t)num_pages * num_kv_heads * page_size >= ((int64_t)1 << 31))
      return SINK_ATTN_ERR_UNSUPPORTED;
  }
  const int cmax = sa::decode_max_chunks(max_seq_len, window, kv_chunk);
  const size_t need = workspace_bytes_for(batch, num_q_heads, head_dim, cmax);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return SINK_ATTN_ERR_WORKSPACE;

  sa::DecodeLaunch a{};
  if (has_cache) {
    const uint64_t rows = (uint64_t)num_pages * num_kv_heads * page_size;
    const bool ok = fp8 ? encode_2d_u8(&a.tm_k, k_cache, head_dim, rows, 16) &&
                              encode_2d_u8(&a.tm_v, v_cache, head_dim, rows, 16)
                        : encode_2d(&a.tm_k, k_cache, head_dim, rows, 16) &&
                              encode_2d(&a.tm_v, v_cache, head_dim, rows, 16);
    if (!ok) return SINK_ATTN_ERR_CUDA;
  } else {
    // No position can be read: the maps are passed but never used.
    memset(&a.tm_k, 0, sizeof a.tm_k);
    memset(&a.tm_v, 0, sizeof a.tm_v);
  }
  a.err = device_error_word();
  if (!a.err) return SINK_ATTN_ERR_CUDA;
  a.q = q;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.sinks = sinks;
  a.k_scale = fp8 ? k_scale : nullptr;
  a.v_scale = fp8 ? v_scale : nullptr;
  a.fp8 = fp8;
  a.out = out;
  a.lse = lse;
  a.o_part = need > 0 ? static_cast<float*>(workspace) : nullptr;
  a.lse_part =
      need > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          align_up((size_t)batch * num_q_heads * cmax * head_dim * 4,
                                                   256))
               : nullptr;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.batch = batch;
  a.max_seq_len = max_seq_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.window = window;
  a.kv_chunk = kv_chunk;
  a.cmax = cmax;
  a.scale = scale;
  a.timeout_ns = g_decode_wait_ns.load();
  a.drain_ns = kWaitTimeoutNs;
  a.withhold_first_page = g_decode_withhold.load();
  return sa::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

sink_attn_status sink_attn_prefill(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                   const sink_attn_bf16* v, const float* sinks,
                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                   int32_t total_tokens, int32_t max_seqlen,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t window, float scale, sink_attn_bf16* out,
                                   sink_attn_stream_t stream) {
  return prefill_impl(q, k, v, sinks, cu_seqlens, num_seqs, total_tokens, max_seqlen,
                      num_q_heads, num_kv_heads, head_dim, window, scale, out, nullptr, stream);
}

sink_attn_status sink_attn_prefill_lse(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                       const sink_attn_bf16* v, const float* sinks,
                                       const int32_t* cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_seqlen,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t window, float scale,
                                       sink_attn_bf16* out, float* lse,
                                       sink_attn_stream_t stream) {
  if (!lse && num_seqs > 0 && total_tokens > 0 && max_seqlen > 0) return SINK_ATTN_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, sinks, cu_seqlens, num_seqs, total_tokens, max_seqlen,
                      num_q_heads, num_kv_heads, head_dim, window, scale, out, lse, stream);
}

sink_attn_status sink_attn_prefill_varlen(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                          const sink_attn_bf16* v, const float* sinks,
                                          const int32_t* cu_seqlens_q,
                                          const int32_t* cu_seqlens_k, int32_t num_seqs,
                                          int32_t total_q, int32_t total_k, int32_t max_seqlen_q,
                                          int32_t max_seqlen_k, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t window,
                                          float scale, sink_attn_bf16* out, float* lse,
                                          sink_attn_stream_t stream) {
  if (!cu_seqlens_k && num_seqs > 0 && total_q > 0 && max_seqlen_q > 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, sinks, cu_seqlens_q, num_seqs, total_q, max_seqlen_q, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, stream, cu_seqlens_k,
                      total_k, max_seqlen_k);
}

size_t sink_attn_prefill_from_host_scratch_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t n_ranges) {
  if (num_seqs < 0 || num_q_heads <= 0 || n_ranges <= 0) return 0;
  return from_host_scratch_bytes(num_seqs, num_q_heads, n_ranges);
}

sink_attn_status sink_attn_prefill_from_host(
    const sink_attn_bf16* q_host, const sink_attn_bf16* k_host, const sink_attn_bf16* v_host,
    const float* sinks_host, const int32_t* cu_seqlens_host, int32_t num_seqs,
    int32_t total_tokens, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t window, float scale, sink_attn_bf16* out_host, sink_attn_bf16* q_dev,
    sink_attn_bf16* k_dev, sink_attn_bf16* v_dev, sink_attn_bf16* out_dev, void* scratch,
    size_t scratch_bytes, int32_t n_ranges, sink_attn_stream_t stream,
    sink_attn_stream_t copy_in, sink_attn_stream_t copy_out) {
  if (num_seqs < 0 || total_tokens < 0 || n_ranges <= 0 || !cu_seqlens_host)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  // The row offsets are host memory here: check them before anything is issued.
  const int32_t* cu = cu_seqlens_host;
  if (cu[0] < 0 || cu[num_seqs] > total_tokens) return SINK_ATTN_ERR_INVALID_ARG;
  for (int s = 0; s < num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return SINK_ATTN_ERR_INVALID_ARG;
  const int32_t lo = cu[0], hi = cu[num_seqs];
  if (num_seqs == 0 || hi == lo) return SINK_ATTN_OK;
  if (!q_host || !k_host || !v_host || !out_host || !q_dev || !k_dev || !v_dev || !out_dev ||
      !scratch)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) || !aligned16(out_dev) ||
      !aligned16(scratch))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (scratch_bytes < from_host_scratch_bytes(num_seqs, num_q_heads, n_ranges))
    return SINK_ATTN_ERR_WORKSPACE;

  // Equal row ranges, in order, across sequence boundaries. Range g: rows [r0, r1) of
  // sequences sa .. sb-1; its queries are those rows and each sequence's keys run from the
  // sequence's first row (earlier ranges have brought those rows in).
  struct Range {
    int32_t r0, r1, sa, sb, mq, mk;
    size_t off;  // int32 offset of its query offsets in the scratch (key offsets follow)
  };
  const int32_t n = std::min<int32_t>(n_ranges, hi - lo);
  std::vector<Range> ranges;
  std::vector<int32_t> host;  // every range's offsets, then the sinks' bits
  ranges.reserve(n);
  int s = 0;
  for (int g = 0; g < n; ++g) {
    Range r{};
    r.r0 = lo + (int32_t)((int64_t)(hi - lo) * g / n);
    r.r1 = lo + (int32_t)((int64_t)(hi - lo) * (g + 1) / n);
    if (r.r1 <= r.r0) continue;
    while (cu[s + 1] <= r.r0) ++s;
    int e = s;
    while (cu[e + 1] < r.r1) ++e;
    r.sa = s;
    r.sb = e + 1;
    r.off = host.size();
    int32_t acc = 0;
    host.push_back(0);
    for (int t = r.sa; t < r.sb; ++t) {
      const int32_t nq = std::min(r.r1, cu[t + 1]) - std::max(r.r0, cu[t]);
      acc += nq;
      host.push_back(acc);
      r.mq = std::max(r.mq, nq);
      r.mk = std::max(r.mk, std::min(r.r1, cu[t + 1]) - cu[t]);
    }
    host.push_back(0);
    for (int t = r.sa; t < r.sb; ++t) host.push_back(std::min(r.r1, cu[t + 1]) - cu[r.sa]);
    ranges.push_back(r);
  }
  const size_t sink_off = host.size();
  if (sinks_host) {
    host.resize(sink_off + num_q_heads);
    memcpy(host.data() + sink_off, sinks_host, sizeof(float) * num_q_heads);
  }

  cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t s_in = copy_in ? reinterpret_cast<cudaStream_t>(copy_in) : main;
  cudaStream_t s_out = copy_out ? reinterpret_cast<cudaStream_t>(copy_out) : main;
  cudaEvent_t ev[4] = {};  // start, input ready, output ready, copies done
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      for (auto& x : ev)
        if (x) cudaEventDestroy(x);
      return SINK_ATTN_ERR_CUDA;
    }
  // An event is captured by each wait when the wait is issued, so one event per role
  // serves every range.
  auto handoff = [&](cudaEvent_t e, cudaStream_t from, cudaStream_t to) {
    if (from == to) return cudaSuccess;
    cudaError_t r = cudaEventRecord(e, from);
    return r == cudaSuccess ? cudaStreamWaitEvent(to, e, 0) : r;
  };
  int32_t* sc = static_cast<int32_t*>(scratch);
  const size_t q_row = (size_t)num_q_heads * head_dim, kv_row = (size_t)num_kv_heads * head_dim;
  sink_attn_status st = SINK_ATTN_OK;
  // The device buffers and the scratch may still be in use by earlier work on `stream`.
  cudaError_t ce = handoff(ev[0], main, s_in);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(sc, host.data(), host.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                         s_in);
  for (size_t g = 0; ce == cudaSuccess && st == SINK_ATTN_OK && g < ranges.size(); ++g) {
    const Range& r = ranges[g];
    const size_t rows = r.r1 - r.r0;
    ce = cudaMemcpyAsync(q_dev + r.r0 * q_row, q_host + r.r0 * q_row, rows * q_row * 2,
                         cudaMemcpyHostToDevice, s_in);
    if (ce == cudaSuccess)
      ce = cudaMemcpyAsync(k_dev + r.r0 * kv_row, k_host + r.r0 * kv_row, rows * kv_row * 2,
                           cudaMemcpyHostToDevice, s_in);
    if (ce == cudaSuccess)
      ce = cudaMemcpyAsync(v_dev + r.r0 * kv_row, v_host + r.r0 * kv_row, rows * kv_row * 2,
                           cudaMemcpyHostToDevice, s_in);
    if (ce == cudaSuccess) ce = handoff(ev[1], s_in, main);
    if (ce != cudaSuccess) break;
    const int32_t ns = r.sb - r.sa, k0 = cu[r.sa];
    st = prefill_impl(q_dev + r.r0 * q_row, k_dev + (size_t)k0 * kv_row,
                      v_dev + (size_t)k0 * kv_row,
                      sinks_host ? reinterpret_cast<const float*>(sc + sink_off) : nullptr,
                      sc + r.off, ns, (int32_t)rows, r.mq, num_q_heads, num_kv_heads, head_dim,
                      window, scale, out_dev + r.r0 * q_row, nullptr, stream,
                      sc + r.off + ns + 1, r.r1 - k0, r.mk);
    if (st != SINK_ATTN_OK) break;
    ce = handoff(ev[2], main, s_out);
    if (ce == cudaSuccess)
      ce = cudaMemcpyAsync(out_host + r.r0 * q_row, out_dev + r.r0 * q_row, rows * q_row * 2,
                           cudaMemcpyDeviceToHost, s_out);
  }
  if (ce == cudaSuccess) ce = handoff(ev[3], s_out, main);  // `stream` orders after the copies
  for (auto& e : ev) cudaEventDestroy(e);  // released once the device has passed them
  if (st != SINK_ATTN_OK) return st;
  return ce == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_decode(const sink_attn_bf16* q, const sink_attn_bf16* k_cache,
                                  const sink_attn_bf16* v_cache, int32_t num_pages,
                                  int32_t page_size, const int32_t* page_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens,
                                  int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, const float* sinks,
                                  int32_t window, float scale, int32_t kv_chunk, void* workspace,
                                  size_t workspace_bytes, sink_attn_bf16* out,
                                  sink_attn_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, nullptr, nullptr, num_pages, page_size, page_table,
                     max_pages_per_seq, seq_lens, batch, max_seq_len, num_q_heads, num_kv_heads,
                     head_dim, sinks, window, scale, kv_chunk, workspace, workspace_bytes, out,
                     nullptr, stream);
}

sink_attn_status sink_attn_decode_lse(const sink_attn_bf16* q, const sink_attn_bf16* k_cache,
                                      const sink_attn_bf16* v_cache, int32_t num_pages,
                                      int32_t page_size, const int32_t* page_table,
                                      int32_t max_pages_per_seq, const int32_t* seq_lens,
                                      int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, const float* sinks,
                                      int32_t window, float scale, int32_t kv_chunk,
                                      void* workspace, size_t workspace_bytes,
                                      sink_attn_bf16* out, float* lse,
                                      sink_attn_stream_t stream) {
  if (!lse && batch > 0) return SINK_ATTN_ERR_INVALID_ARG;
  return decode_impl(q, k_cache, v_cache, nullptr, nullptr, num_pages, page_size, page_table,
                     max_pages_per_seq, seq_lens, batch, max_seq_len, num_q_heads, num_kv_heads,
                     head_dim, sinks, window, scale, kv_chunk, workspace, workspace_bytes, out, lse,
                     stream);
}

}  // extern "C"

namespace {

// Shared argument checks of the paged entry points; fills everything but the kernels'
// own fields. Returns SINK_ATTN_OK when a launch should follow.
// k_cache/v_cache: bf16 pages, or (k_scale non-null) e4m3 code pages with row scales.
sink_attn_status append_args(const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
                             void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                             int32_t num_pages,
                             int32_t page_size, const int32_t* page_table,
                             int32_t max_pages_per_seq, const int32_t* cu_seqlens,
                             const int32_t* seq_lens, int32_t num_seqs, int32_t total_tokens,
                             int32_t num_kv_heads, int32_t head_dim, sa::AppendLaunch& a) {
  if (num_seqs < 0 || total_tokens < 0 || num_pages < 0 || max_pages_per_seq < 0 ||
      num_kv_heads <= 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (page_size != 16) return SINK_ATTN_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !cu_seqlens || !seq_lens)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned4(page_table) || !aligned4(cu_seqlens) || !aligned4(seq_lens))
    return SINK_ATTN_ERR_INVALID_ARG;
  const bool fp8 = k_scale != nullptr || v_scale != nullptr;
  if (fp8 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || max_pages_per_seq <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if ((int64_t)num_pages * num_kv_heads * page_size >= ((int64_t)1 << 31) ||
      (int64_t)total_tokens * num_kv_heads >= ((int64_t)1 << 31))
    return SINK_ATTN_ERR_UNSUPPORTED;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = fp8 ? nullptr : static_cast<uint16_t*>(k_cache);
  a.v_cache = fp8 ? nullptr : static_cast<uint16_t*>(v_cache);
  a.k_codes = fp8 ? static_cast<uint8_t*>(k_cache) : nullptr;
  a.v_codes = fp8 ? static_cast<uint8_t*>(v_cache) : nullptr;
  a.k_scale = fp8 ? k_scale : nullptr;
  a.v_scale = fp8 ? v_scale : nullptr;
  a.page_table = page_table;
  a.cu_seqlens = cu_seqlens;
  a.kv_lens = seq_lens;
  a.err = device_error_word();
  if (!a.err) return SINK_ATTN_ERR_CUDA;
  a.num_seqs = num_seqs;
  a.total_tokens = total_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_pages = num_pages;
  a.max_pages = max_pages_per_seq;
  return SINK_ATTN_OK;
}

}  // namespace

extern "C" {

sink_attn_status sink_attn_append_kv(const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
                                     sink_attn_bf16* k_cache, sink_attn_bf16* v_cache,
                                     int32_t num_pages, int32_t page_size,
                                     const int32_t* page_table, int32_t max_pages_per_seq,
                                     const int32_t* cu_seqlens, const int32_t* seq_lens,
                                     int32_t num_seqs, int32_t total_tokens, int32_t num_kv_heads,
                                     int32_t head_dim, sink_attn_stream_t stream) {
  if (num_seqs == 0 || total_tokens == 0) {
    return (num_seqs < 0 || total_tokens < 0) ? SINK_ATTN_ERR_INVALID_ARG : SINK_ATTN_OK;
  }
  sa::AppendLaunch a{};
  const sink_attn_status st =
      append_args(k_new, v_new, k_cache, v_cache, nullptr, nullptr, num_pages, page_size, page_table,
                  max_pages_per_seq, cu_seqlens, seq_lens, num_seqs, total_tokens, num_kv_heads,
                  head_dim, a);
  if (st != SINK_ATTN_OK) return st;
  return sa::launch_append_kv(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_prefill_paged(
    const sink_attn_bf16* q, const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
    sink_attn_bf16* k_cache, sink_attn_bf16* v_cache, int32_t num_pages, int32_t page_size,
    const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* cu_seqlens,
    const int32_t* seq_lens, int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
    int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    const float* sinks, int32_t window, float scale, sink_attn_bf16* out, float* lse,
    sink_attn_stream_t stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_q_len < 0 || max_seq_len < 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return SINK_ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_tokens == 0 || max_q_len == 0) return SINK_ATTN_OK;
  if (!q || !out) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (sinks && !aligned4(sinks)) || (lse && !aligned4(lse)))
    return SINK_ATTN_ERR_INVALID_ARG;
  if ((int64_t)total_tokens * num_q_heads >= ((int64_t)1 << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  const int64_t n_qt = (max_q_len + 127) / 128;
  if (n_qt * num_seqs * num_q_heads >= ((int64_t)1 << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  sa::AppendLaunch ap{};
  sink_attn_status st =
      append_args(k_new, v_new, k_cache, v_cache, nullptr, nullptr, num_pages, page_size, page_table,
                  max_pages_per_seq, cu_seqlens, seq_lens, num_seqs, total_tokens, num_kv_heads,
                  head_dim, ap);
  if (st != SINK_ATTN_OK) return st;

  sa::PrefillLaunch a{};
  const uint64_t rows = (uint64_t)num_pages * num_kv_heads * page_size;
  if (!encode_3d(&a.tm_q, q, head_dim, num_q_heads, total_tokens, 128) ||
      !encode_2d(&a.tm_k, k_cache, head_dim, rows, 16) ||
      !encode_2d(&a.tm_v, v_cache, head_dim, rows, 16))
    return SINK_ATTN_ERR_CUDA;
  a.err = ap.err;
  a.num_sms = num_sms_current();
  if (a.num_sms <= 0) return SINK_ATTN_ERR_CUDA;
  a.cu_seqlens = cu_seqlens;
  a.kv_lens = seq_lens;
  a.page_table = page_table;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.max_kv = max_seq_len;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.num_seqs = num_seqs;
  a.total_tokens = total_tokens;
  a.max_seqlen = max_q_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.window = window;
  a.scale = scale;
  a.timeout_ns = kWaitTimeoutNs;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (sa::launch_append_kv(ap, s) != cudaSuccess) return SINK_ATTN_ERR_CUDA;
  return sa::launch_prefill(a, s) == cudaSuccess ? SINK_ATTN_OK : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_merge_states(const sink_attn_bf16* o_a, const float* lse_a,
                                        const sink_attn_bf16* o_b, const float* lse_b,
                                        int32_t rows, int32_t num_heads, int32_t head_dim,
                                        sink_attn_bf16* o_out, float* lse_out,
                                        sink_attn_stream_t stream) {
  if (rows < 0 || num_heads <= 0) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return SINK_ATTN_OK;
  if ((int64_t)rows * num_heads >= ((int64_t)1 << 31)) return SINK_ATTN_ERR_UNSUPPORTED;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out) return SINK_ATTN_ERR_INVALID_ARG;
  if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o_out) || !aligned4(lse_a) ||
      !aligned4(lse_b) || (lse_out && !aligned4(lse_out)))
    return SINK_ATTN_ERR_INVALID_ARG;
  sa::MergeLaunch a;
  a.o_a = o_a;
  a.lse_a = lse_a;
  a.o_b = o_b;
  a.lse_b = lse_b;
  a.o_out = o_out;
  a.lse_out = lse_out;
  a.rows = rows;
  a.heads = num_heads;
  a.head_dim = head_dim;
  return sa::launch_merge_states(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_quantize_fp8(const sink_attn_bf16* x, int64_t rows, int32_t head_dim,
                                        uint8_t* codes, float* scales,
                                        sink_attn_stream_t stream) {
  if (rows < 0) return SINK_ATTN_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SINK_ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return SINK_ATTN_OK;
  if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes) || !aligned4(scales))
    return SINK_ATTN_ERR_INVALID_ARG;
  if (rows >= ((int64_t)1 << 34)) return SINK_ATTN_ERR_UNSUPPORTED;
  sa::QuantizeLaunch a;
  a.x = x;
  a.codes = codes;
  a.scales = scales;
  a.rows = rows;
  a.head_dim = head_dim;
  return sa::launch_quantize_fp8(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_append_kv_fp8(const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
                                         uint8_t* k_codes, uint8_t* v_codes, float* k_scale,
                                         float* v_scale, int32_t num_pages, int32_t page_size,
                                         const int32_t* page_table, int32_t max_pages_per_seq,
                                         const int32_t* cu_seqlens, const int32_t* seq_lens,
                                         int32_t num_seqs, int32_t total_tokens,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         sink_attn_stream_t stream) {
  if (num_seqs == 0 || total_tokens == 0) {
    return (num_seqs < 0 || total_tokens < 0) ? SINK_ATTN_ERR_INVALID_ARG : SINK_ATTN_OK;
  }
  if (!k_scale || !v_scale) return SINK_ATTN_ERR_INVALID_ARG;
  sa::AppendLaunch a{};
  const sink_attn_status st =
      append_args(k_new, v_new, k_codes, v_codes, k_scale, v_scale, num_pages, page_size,
                  page_table, max_pages_per_seq, cu_seqlens, seq_lens, num_seqs, total_tokens,
                  num_kv_heads, head_dim, a);
  if (st != SINK_ATTN_OK) return st;
  return sa::launch_append_kv(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SINK_ATTN_OK
             : SINK_ATTN_ERR_CUDA;
}

sink_attn_status sink_attn_decode_fp8(const sink_attn_bf16* q, const uint8_t* k_codes,
                                      const uint8_t* v_codes, const float* k_scale,
                                      const float* v_scale, int32_t num_pages, int32_t page_size,
                                      const int32_t* page_table, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      const float* sinks, int32_t window, float scale,
                                      int32_t kv_chunk, void* workspace, size_t workspace_bytes,
                                      sink_attn_bf16* out, float* lse,
                                      sink_attn_stream_t stream) {
  if (batch > 0 && max_seq_len > 0 && (!k_scale || !v_scale)) return SINK_ATTN_ERR_INVALID_ARG;
  // With no cache position at all the bf16 path writes the zero outputs the same way.
  const bool any = batch > 0 && max_seq_len > 0;
  return decode_impl(q, k_codes, v_codes, any ? k_scale : nullptr, any ? v_scale : nullptr,
                     num_pages, page_size, page_table, max_pages_per_seq, seq_lens, batch,
                     max_seq_len, num_q_heads, num_kv_heads, head_dim, sinks, window, scale,
                     kv_chunk, workspace, workspace_bytes, out, lse, stream);
}

sink_attn_status sink_attn_read_device_error(sink_attn_stream_t stream, uint32_t* bits_out) {
  if (bits_out) *bits_out = 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SINK_ATTN_ERR_CUDA;
  unsigned* p = device_error_word();
  if (!p) return SINK_ATTN_ERR_CUDA;
  unsigned bits = 0;
  const unsigned zero = 0;
  if (cudaMemcpy(&bits, p, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return SINK_ATTN_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  return bits ? SINK_ATTN_ERR_DEVICE : SINK_ATTN_OK;
}

}  // extern "C"
