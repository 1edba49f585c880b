// kv_append.cu — write the K/V rows of newly processed tokens into the paged HND cache
// ("Qwen hosten op Blackwell", §Prefillers / §Inzet op GB200 NVL72: prefill fills the KV
// cache, laid out head-major with tokens contiguous per (page, kv head)).
//
// Sequence s owns new rows [cu[s], cu[s+1]) of k_new/v_new; after the append it holds
// kv_lens[s] tokens, the new rows being its last ones: row cu[s] + i goes to position
// kv_lens[s] - n_s + i, i.e. page page_table[s][pos / 16], slot pos % 16. A bf16 cache
// takes one warp per new row, moving its K and V rows of every kv head as 16-byte chunks.
// Rows of no sequence, inconsistent lengths and page ids outside [0, num_pages) are
// skipped and recorded.
//
// FP8 cache: the warp quantises each row on the way (e4m3 codes plus one fp32 scale per
// row; the 8-bit direction of "Qwen hosten op Blackwell", §Kwantisering):
//   amax = max |x|,  scale = amax / 448,  code = e4m3_rn_satfinite(x * (448 / amax)),
// every operation an IEEE fp32 operation rounded to nearest, so the row's largest element
// becomes +-448; a zero row has scale 0 and zero codes. The same quantiser converts
// contiguous rows (an existing bf16 cache, for instance).
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

// Quantise one bf16 row of D elements held by a warp (D/32 consecutive elements per lane):
// writes the lane's codes and, from lane 0, the row scale.
template <int D>
__device__ __forceinline__ void quantize_row(const uint16_t* src, uint8_t* codes, float* scale,
                                             int lane) {
  constexpr int E = D / 32;  // 2 or 4
  float x[E];
  if constexpr (E == 2) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(src)[lane];
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    x[0] = f.x;
    x[1] = f.y;
  } else {
    const uint2 w = reinterpret_cast<const uint2*>(src)[lane];
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    x[0] = f0.x;
    x[1] = f0.y;
    x[2] = f1.x;
    x[3] = f1.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 y = make_float2(__fmul_rn(x[e], inv), __fmul_rn(x[e + 1], inv));
    packed |= (uint32_t)__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3) << (8 * e);
  }
  if constexpr (E == 2) {
    reinterpret_cast<uint16_t*>(codes)[lane] = (uint16_t)packed;
  } else {
    reinterpret_cast<uint32_t*>(codes)[lane] = packed;
  }
  if (lane == 0) *scale = __fdiv_rn(amax, 448.f);
}

template <int D>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const QuantizeLaunch a) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= a.rows) return;
  quantize_row<D>(a.x + r * D, a.codes + r * D, a.scales + r, threadIdx.x & 31);
}

// FP8 cache: one warp per (new row, kv head), quantising the row on the way.
template <int D>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const AppendLaunch a) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)a.total_tokens * a.num_kv_heads) return;
  const int r = (int)(wid / a.num_kv_heads), g = (int)(wid - (long long)r * a.num_kv_heads);
  if (r < a.cu_seqlens[0] || r >= a.cu_seqlens[a.num_seqs]) return;  // row of no sequence
  int lo = 0, hi = a.num_seqs;  // the sequence s with cu[s] <= r < cu[s+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.cu_seqlens[mid] <= r) lo = mid; else hi = mid;
  }
  const int s = lo;
  const int n = a.cu_seqlens[s + 1] - a.cu_seqlens[s];
  const int L = a.kv_lens[s];
  if (n < 0 || L < n || (L + 15) / 16 > a.max_pages) {
    if (lane == 0) atomicOr(a.err, kErrSeqLen);
    return;
  }
  const int pos = L - n + (r - a.cu_seqlens[s]);
  const int pid = a.page_table[(size_t)s * a.max_pages + pos / 16];
  if (pid < 0 || pid >= a.num_pages) {
    if (lane == 0) atomicOr(a.err, kErrPageId);
    return;
  }
  const size_t src = ((size_t)r * a.num_kv_heads + g) * D;
  const size_t slot = ((size_t)pid * a.num_kv_heads + g) * 16 + pos % 16;
  const size_t dst = slot * D;
  quantize_row<D>(a.k_new + src, a.k_codes + dst, a.k_scale + slot, lane);
  quantize_row<D>(a.v_new + src, a.v_codes + dst, a.v_scale + slot, lane);
}

// bf16 cache: one warp per new row, all kv heads. The row's lookups (its sequence, the
// sequence's length, the page id) are dependent global loads; paying them once per row
// instead of once per (row, kv head), with every lane copying, took the chunked gpt-oss
// prefill's append (8192 rows x 8 kv heads) from 15 to 8.5 us.
template <int D>
__global__ void __launch_bounds__(256) kv_append_rows_kernel(const AppendLaunch a) {
  const long long r64 = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r64 >= a.total_tokens) return;
  const int r = (int)r64;
  if (r < a.cu_seqlens[0] || r >= a.cu_seqlens[a.num_seqs]) return;  // row of no sequence
  int lo = 0, hi = a.num_seqs;  // the sequence s with cu[s] <= r < cu[s+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.cu_seqlens[mid] <= r) lo = mid; else hi = mid;
  }
  const int s = lo;
  const int n = a.cu_seqlens[s + 1] - a.cu_seqlens[s];
  const int L = a.kv_lens[s];
  if (n < 0 || L < n || (L + 15) / 16 > a.max_pages) {
    if (lane == 0) atomicOr(a.err, kErrSeqLen);
    return;
  }
  const int pos = L - n + (r - a.cu_seqlens[s]);
  const int pid = a.page_table[(size_t)s * a.max_pages + pos / 16];
  if (pid < 0 || pid >= a.num_pages) {
    if (lane == 0) atomicOr(a.err, kErrPageId);
    return;
  }
  constexpr int kChunks = D / 8;               // 16-byte chunks per (row, kv head)
  const int per = a.num_kv_heads * kChunks;    // chunks of the row's K (or V), all heads
  const uint4* ksrc = reinterpret_cast<const uint4*>(a.k_new + (size_t)r * a.num_kv_heads * D);
  const uint4* vsrc = reinterpret_cast<const uint4*>(a.v_new + (size_t)r * a.num_kv_heads * D);
  const size_t slot0 = (size_t)pid * a.num_kv_heads * 16 + pos % 16;  // kv head 0's slot
  for (int c = lane; c < 2 * per; c += 32) {
    const bool v = c >= per;
    const int cc = v ? c - per : c;
    const int g = cc / kChunks, ch = cc - g * kChunks;
    const uint4 x = (v ? vsrc : ksrc)[cc];
    uint4* dst = reinterpret_cast<uint4*>((v ? a.v_cache : a.k_cache) + (slot0 + (size_t)g * 16) * D);
    dst[ch] = x;
  }
}

}  // namespace

cudaError_t launch_append_kv(const AppendLaunch& a, cudaStream_t stream) {
  const long long warps = (long long)a.total_tokens * a.num_kv_heads;
  if (warps <= 0 || a.num_seqs <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  const unsigned row_blocks = (unsigned)(((long long)a.total_tokens + 7) / 8);
  const bool f8 = a.k_codes != nullptr;
  if (a.head_dim == 64) {
    if (f8) kv_append_fp8_kernel<64><<<blocks, 256, 0, stream>>>(a);
    else kv_append_rows_kernel<64><<<row_blocks, 256, 0, stream>>>(a);
  } else {
    if (f8) kv_append_fp8_kernel<128><<<blocks, 256, 0, stream>>>(a);
    else kv_append_rows_kernel<128><<<row_blocks, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const QuantizeLaunch& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((a.rows + 7) / 8);
  if (a.head_dim == 64) {
    quantize_rows_kernel<64><<<blocks, 256, 0, stream>>>(a);
  } else {
    quantize_rows_kernel<128><<<blocks, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sa
