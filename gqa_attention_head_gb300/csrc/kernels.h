// kernels.h — internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

struct PrefillLaunch {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps {head_dim, heads, tokens}, box {64, 1, 128};
                                 // paged: tm_k/tm_v 2-D over the cache, box {64, 16}
  const int32_t* cu_seqlens;     // query rows (contiguous: also key rows)
  const int32_t* kv_lens;        // paged: keys per sequence after the append; null otherwise
  const int32_t* cu_seqlens_k;   // contiguous K/V with their own rows: [num_seqs + 1]; or null
  int total_k;                   // with cu_seqlens_k: rows of K and V
  const int32_t* page_table;     // paged: [num_seqs][max_pages]
  int max_pages, num_pages, max_kv;
  const float* sinks;            // nullable
  void* out;                     // bf16 [T, Hq, D]
  float* lse;                    // fp32 [T, Hq] natural log, or null
  unsigned* err;                 // device error word
  int num_seqs, total_tokens, max_seqlen, num_q_heads, num_kv_heads, head_dim, window;
  float scale;
  int num_sms;
  uint64_t timeout_ns;
  int band;                      // the short-window kernel: tm_q has box {64, 8, 16} and
                                 // tm_k/tm_v box {64, 1, 160} (prefill_band_applies)
  CUtensorMap tm_o;              // band: `out` as {head_dim, heads, tokens}, box {64, 8, 4}
};

// The short-window prefill kernel (prefill_band.cu): 32 queries x 8 query heads per unit
// (two head tiles of 16 queries x 8 heads), each unit reading one 160-key span. It serves contiguous head_dim-64 calls with a window
// of 1..128 keys when every kv head has a multiple of 8 query heads, up to kBandMaxSeqs
// sequences and kBandMaxUnits units per CTA (bounded here from the row count).
constexpr int kBandMaxSeqs = 1024;
constexpr int kBandMaxUnits = 512;
inline bool prefill_band_applies(int head_dim, int window, int num_q_heads, int num_kv_heads,
                                 long long total_tokens, int num_seqs, int num_sms) {
  if (head_dim != 64 || window <= 0 || window > 128 || num_sms <= 0) return false;
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  if (g % 8 != 0 || num_seqs <= 0 || num_seqs > kBandMaxSeqs) return false;
  const long long blocks = total_tokens / 32 + num_seqs;  // query blocks of 32, at most
  return blocks * num_kv_heads * (g / 8) <= (long long)kBandMaxUnits * num_sms;
}

struct DecodeLaunch {
  CUtensorMap tm_k, tm_v;        // 2-D maps {head_dim, pages*Hkv*page_size}, box {64, 16};
                                 // FP8: uint8 maps, box {head_dim, 16}
  const float* k_scale;          // FP8: [pages, Hkv, page_size] fp32 row scales; else null
  const float* v_scale;
  bool fp8;
  const void* q;                 // bf16 [B, Hq, D]
  const int32_t* page_table;
  const int32_t* seq_lens;
  const float* sinks;            // nullable
  void* out;                     // bf16 [B, Hq, D]
  float* lse;                    // fp32 [B, Hq] natural log, or null
  float* o_part;                 // [B, Hq, Cmax, D]   (null when Cmax == 1)
  float* lse_part;               // [B, Hq, Cmax]
  unsigned* err;
  int num_pages, page_size, max_pages, batch, max_seq_len, num_q_heads, num_kv_heads, head_dim,
      window, kv_chunk, cmax;
  float scale;
  uint64_t timeout_ns;           // limit of every pipeline wait
  uint64_t drain_ns;             // limit of the teardown waits for copies still in flight
  int withhold_first_page;       // test switch: never copy page 0 of (chunk 0, kv head 0,
                                 // sequence 0), so that its consumers' waits run out
};

// Number of split-KV chunks the grid provides for (window-limited visible range).
inline int decode_max_chunks(int max_seq_len, int window, int kv_chunk) {
  long vis = max_seq_len;
  if (window > 0 && window < vis) vis = window;
  long c = (vis + kv_chunk - 1) / kv_chunk;
  return c < 1 ? 1 : (int)c;
}

struct MergeLaunch {
  const void* o_a;               // bf16 [rows, heads, D]
  const float* lse_a;            // fp32 [rows, heads]
  const void* o_b;
  const float* lse_b;
  void* o_out;                   // bf16 [rows, heads, D]
  float* lse_out;                // fp32 [rows, heads] or null
  int rows, heads, head_dim;
};

struct AppendLaunch {
  const uint16_t* k_new;         // bf16 bits [T, Hkv, D]
  const uint16_t* v_new;
  uint16_t* k_cache;             // bf16 bits [pages, Hkv, 16, D] (null for an FP8 cache)
  uint16_t* v_cache;
  uint8_t* k_codes;              // FP8 cache: e4m3 [pages, Hkv, 16, D] (null for bf16)
  uint8_t* v_codes;
  float* k_scale;                // FP8 cache: [pages, Hkv, 16] row scales
  float* v_scale;
  const int32_t* page_table;     // [num_seqs][max_pages]
  const int32_t* cu_seqlens;     // [num_seqs + 1] new rows
  const int32_t* kv_lens;        // [num_seqs] tokens after the append
  unsigned* err;
  int num_seqs, total_tokens, num_kv_heads, head_dim, num_pages, max_pages;
};

struct QuantizeLaunch {
  const uint16_t* x;             // bf16 bits [rows, D]
  uint8_t* codes;                // e4m3 [rows, D]
  float* scales;                 // [rows]
  long long rows;
  int head_dim;
};

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream);
cudaError_t launch_prefill_band(const PrefillLaunch& a, cudaStream_t stream);
cudaError_t launch_quantize_fp8(const QuantizeLaunch& a, cudaStream_t stream);
cudaError_t launch_append_kv(const AppendLaunch& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream);
cudaError_t launch_merge_states(const MergeLaunch& a, cudaStream_t stream);

}  // namespace sa
