/*
 * sink_attn.h — C ABI of the GB300 (sm_103a) sink-attention library.
 *
 * The operation: grouped-query attention (GQA) in which every query head h owns
 * one learned scalar, its sink logit sink[h], that takes part in the softmax as
 * one extra logit with no value row
 *   ("GPT-OSS am Day 0", §GPT-OSS auf Hopper, item "Attention: GQA mit
 *    Attention-Sinks": every attention head has a pre-trained sink parameter
 *    that enters the softmax;
 *    §Kernel für GPT-OSS › Sink-Attention ¶1: an extra bias term before the
 *    softmax, accumulated next to the Q·K products).
 *
 * For query row i of query head h, with key/value head g = floor(h / G),
 * G = num_q_heads / num_kv_heads, and the set V(i) of keys row i may see:
 *
 *     s_ij   = scale * <q_i, k_j>                       for j in V(i)
 *     m      = max(sink[h], max_j s_ij)
 *     Z      = exp(sink[h] - m) + sum_j exp(s_ij - m)
 *     out_i  = sum_j exp(s_ij - m) * v_j / Z
 *
 * The sink is compared with the *scaled* logits (it is not multiplied by
 * `scale`) and adds to the denominator only. sink[h] = -INFINITY gives plain
 * softmax attention. A row with no visible key and sink = -inf is defined as 0.
 * The equations of the page's section did not survive text extraction; the
 * prose around them (one additive term in the softmax, a running maximum that
 * starts at the sink value, the sink counted in only one chunk of a split along
 * the sequence — §Sink-Attention ¶3) fixes the form above.
 *
 * Visibility (causal, optional sliding window W):
 *   prefill: key j (position inside the same sequence) is visible to query
 *            position i iff  j <= i  and  (W <= 0  or  i - j < W).
 *            A window W > 0 therefore covers exactly W keys, the query's own
 *            position included.
 *   decode:  the single query sits at position L-1 of its sequence (its own
 *            key/value already in the cache); visible keys are the cache
 *            positions [max(0, L - W), L)  (W <= 0: [0, L)).
 *
 * Split-KV decode ("GPT-OSS am Day 0", §Sink-Attention ¶2-¶3): the visible range
 * is cut into chunks of `kv_chunk` tokens that start at its first token; each
 * chunk yields a partial output and log-sum-exp, and only the chunk that starts
 * the visible range carries the sink. A merge kernel combines the chunks.
 *
 * Paged KV cache in HND order ("Qwen hosten op Blackwell", §Inzet op GB200 NVL72:
 * heads lead, tokens contiguous): k_cache and v_cache are separate arrays
 *   [num_pages][num_kv_heads][page_size][head_dim]   (bf16, row-major)
 * so one (page, kv head) block holds page_size consecutive tokens.
 * page_table[b * max_pages_per_seq + p] is the physical page holding tokens
 * [p*page_size, (p+1)*page_size) of sequence b.
 *
 * Entry points
 *   sink_attn_prefill / _prefill_lse     ragged causal prefill (contiguous K/V)
 *   sink_attn_prefill_varlen             the same with more keys than queries per sequence
 *   sink_attn_prefill_from_host          the ragged prefill from and back to host memory,
 *                                        copies and kernels overlapped in row ranges
 *   sink_attn_decode / _decode_lse       paged split-KV decode (bf16 cache)
 *   sink_attn_decode_static_workspace    the decode with library-held scratch
 *   sink_attn_append_kv                  write new K/V rows into the paged cache
 *   sink_attn_prefill_paged              chunked prefill: append, then attend over the cache
 *   sink_attn_merge_states               combine two (output, log-sum-exp) states
 *   sink_attn_quantize_fp8 / _append_kv_fp8 / _decode_fp8   the FP8 (e4m3) cache
 *   sink_attn_decode_workspace_bytes, sink_attn_status_string,
 *   sink_attn_read_device_error, sink_attn_num_sms
 *   sink_attn_debug_decode_withhold_page   test switch for the decode's timeout path
 *
 * Conventions shared by every entry point
 *   - Every pointer is device memory owned by the caller (sink_attn_prefill_from_host
 *     also takes host arrays, named *_host). The library allocates and frees no memory;
 *     decode scratch is the caller's `workspace`. The one exception is
 *     sink_attn_decode_static_workspace, whose scratch is a fixed array inside the
 *     library (reserved when its module is loaded on a device, see there).
 *   - Every call is asynchronous on `stream` and never synchronises the host.
 *     Host-side size arguments (max_seqlen, max_seq_len, total_tokens) exist so
 *     that no device array has to be read back.
 *   - bf16 tensors are passed as `sink_attn_bf16` (the raw 16-bit pattern).
 *   - Output is written out of place; inputs are not modified, except the paged
     cache that sink_attn_append_kv, sink_attn_append_kv_fp8 and
     sink_attn_prefill_paged fill in place (only the appended slots).
 *   - Pointers must be 16-byte aligned; tensors are dense (no strides). A prefill `out`
 *     that is 32-byte aligned (as every CUDA allocation is) is written in whole 32-byte
 *     sectors, which is faster; a 16-byte aligned one gives the same bits.
 *   - Zero-length sequences and batches are legal: their outputs are zero.
 *   - Argument errors are reported before anything is launched and leave every
 *     output untouched.
 *   - Device-side checks (bad page id, inconsistent cu_seqlens / seq_lens, a
 *     pipeline wait that exceeds its time limit) never trap: the kernel records
 *     a bit in a device error word, skips the bad access and returns.
 *     sink_attn_read_device_error() reports and clears that word.
 */
#ifndef SINK_ATTN_H
#define SINK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raw bf16 bit pattern (1 sign, 8 exponent, 7 mantissa bits). */
typedef uint16_t sink_attn_bf16;

/* Layout-compatible with cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* sink_attn_stream_t;

typedef enum sink_attn_status {
  SINK_ATTN_OK = 0,
  SINK_ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hq % Hkv != 0 */
  SINK_ATTN_ERR_UNSUPPORTED = 2, /* head_dim, page_size or group size not built */
  SINK_ATTN_ERR_WORKSPACE = 3,   /* decode workspace missing or too small */
  SINK_ATTN_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  SINK_ATTN_ERR_DEVICE = 5       /* a device-side check fired (see below) */
} sink_attn_status;

/* Bits of the device error word returned through sink_attn_read_device_error. */
#define SINK_ATTN_DEVERR_WAIT_TIMEOUT 0x1u /* a pipeline wait exceeded its limit   */
#define SINK_ATTN_DEVERR_CU_SEQLENS 0x2u   /* cu_seqlens not monotone / past total */
#define SINK_ATTN_DEVERR_PAGE_ID 0x4u      /* page_table entry outside [0,pages)   */
#define SINK_ATTN_DEVERR_SEQ_LEN 0x8u      /* seq_lens[b] < 0 or > max bound       */

/*
 * Ragged causal prefill ("GPT-OSS am Day 0", §Sink-Attention ¶4: one kernel
 * template serves prefill and decode; "Qwen hosten op Blackwell", §Prefillers:
 * prefill is compute-bound).
 *
 *   q          [total_tokens][num_q_heads][head_dim]   bf16
 *   k, v       [total_tokens][num_kv_heads][head_dim]  bf16
 *   sinks      [num_q_heads] fp32, or NULL for no sink (same as all -inf)
 *   cu_seqlens [num_seqs + 1] int32, device; cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[num_seqs] <= total_tokens. Sequence s owns token rows
 *              [cu_seqlens[s], cu_seqlens[s+1]) of q, k, v and out.
 *   max_seqlen host-side upper bound of every sequence length (>= 0). A longer
 *              sequence sets SINK_ATTN_DEVERR_CU_SEQLENS; its rows past the bound
 *              hold unspecified values afterwards (a kernel may or may not write
 *              them).
 *   window     W > 0: sliding window of W keys; W <= 0: full causal.
 *   scale      multiplier of q·k (typically 1/sqrt(head_dim)).
 *   out        [total_tokens][num_q_heads][head_dim] bf16. Rows of tokens that
 *              belong to no sequence are not written.
 *
 *   Supported: head_dim in {64, 128}; any num_q_heads that is a multiple of
 *   num_kv_heads; total_tokens < 2^31 / num_q_heads.
 */
sink_attn_status sink_attn_prefill(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                   const sink_attn_bf16* v, const float* sinks,
                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                   int32_t total_tokens, int32_t max_seqlen,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t window, float scale,
                                   sink_attn_bf16* out, sink_attn_stream_t stream);

/*
 * Paged split-KV decode, one query token per sequence ("GPT-OSS am Day 0",
 * §Sink-Attention ¶2-¶3; "Qwen hosten op Blackwell", §Decoders: decode is
 * memory-bound).
 *
 *   q          [batch][num_q_heads][head_dim] bf16
 *   k_cache,
 *   v_cache    [num_pages][num_kv_heads][page_size][head_dim] bf16 (HND pages)
 *   page_table [batch][max_pages_per_seq] int32, device
 *   seq_lens   [batch] int32, device; 0 <= seq_lens[b] <= max_seq_len and
 *              ceil(seq_lens[b] / page_size) <= max_pages_per_seq.
 *   max_seq_len host-side upper bound of seq_lens (sizes the chunk grid).
 *   sinks      [num_q_heads] fp32 or NULL.
 *   window     W > 0: attend to the last W cache positions; W <= 0: all.
 *   kv_chunk   split length in tokens (> 0, multiple of page_size).
 *   workspace  device scratch of at least
 *              sink_attn_decode_workspace_bytes(batch, num_q_heads, head_dim,
 *              max_seq_len, kv_chunk) bytes, 16-byte aligned; may be NULL when
 *              that size is 0. Its contents need no initialisation and are
 *              meaningless after the call. Two calls in flight at once must not
 *              share a workspace.
 *   out        [batch][num_q_heads][head_dim] bf16
 *
 *   Supported: head_dim in {64, 128}; page_size 16; group size
 *   G = num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}.
 */
sink_attn_status sink_attn_decode(const sink_attn_bf16* q, const sink_attn_bf16* k_cache,
                                  const sink_attn_bf16* v_cache, int32_t num_pages,
                                  int32_t page_size, const int32_t* page_table,
                                  int32_t max_pages_per_seq, const int32_t* seq_lens,
                                  int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, const float* sinks,
                                  int32_t window, float scale, int32_t kv_chunk,
                                  void* workspace, size_t workspace_bytes,
                                  sink_attn_bf16* out, sink_attn_stream_t stream);

/*
 * Allocation-free decode. The pages have no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory: a plugin that only receives
 * input and output pointers from a host framework owning every allocation, or a
 * latency-critical decode loop that must not call cudaMalloc (an allocation can
 * synchronise the device).
 *
 * Same arguments, layouts, validation and results as sink_attn_decode, without
 * `workspace`/`workspace_bytes`: the split-KV scratch is a fixed array inside the
 * library, SINK_ATTN_STATIC_WORKSPACE_BYTES long, reserved on every GPU that loads
 * the library until the process exits. Sizes whose scratch
 * (sink_attn_decode_workspace_bytes with the window applied) exceeds it are rejected
 * with SINK_ATTN_ERR_WORKSPACE before anything is launched. The call itself allocates
 * nothing. The first call on a device looks up the array's device address there
 * (once per device, with that device current). CUDA loads a library's device code
 * lazily by default (CUDA_MODULE_LOADING=LAZY): the module that holds the array is then
 * loaded, and its memory reserved by the driver, during that first lookup, which may
 * allocate and synchronise. So the array is held on every GPU where this entry point
 * has been called (on every GPU that loads the library when loading is eager), and one
 * warm-up call per device belongs before the latency-critical loop and before any
 * stream capture. Every call shares the one array and leaves its contents behind;
 * nothing in it needs to start at zero, but calls that overlap on the GPU (other
 * streams, other threads) race on it: serialise them.
 */
#define SINK_ATTN_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

sink_attn_status sink_attn_decode_static_workspace(
    const sink_attn_bf16* q, const sink_attn_bf16* k_cache, const sink_attn_bf16* v_cache,
    int32_t num_pages, int32_t page_size, const int32_t* page_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, const float* sinks, int32_t window, float scale,
    int32_t kv_chunk, sink_attn_bf16* out, sink_attn_stream_t stream);

/*
 * Append to the paged cache ("Qwen hosten op Blackwell", §Prefillers: prefill fills the
 * HND KV cache that decode reads). Sequence s has new rows [cu_seqlens[s],
 * cu_seqlens[s+1]) of k_new / v_new and, after the append, seq_lens[s] cached tokens,
 * the new rows being its last ones: new row cu_seqlens[s] + i is written to position
 * seq_lens[s] - n_s + i (n_s its number of new rows), i.e. to slot pos % page_size of page
 * page_table[s][pos / page_size].
 *
 *   k_new, v_new [total_tokens][num_kv_heads][head_dim] bf16
 *   k_cache, v_cache [num_pages][num_kv_heads][page_size][head_dim] bf16, written in place
 *   page_table [num_seqs][max_pages_per_seq] int32; cu_seqlens [num_seqs + 1] int32;
 *   seq_lens [num_seqs] int32 (>= n_s, <= max_pages_per_seq * page_size)
 * Positions other than the appended ones are not touched. A page id outside
 * [0, num_pages) or an inconsistent length is skipped and recorded in the device error
 * word (SINK_ATTN_DEVERR_PAGE_ID / _SEQ_LEN). Supported: head_dim in {64, 128},
 * page_size 16.
 */
sink_attn_status sink_attn_append_kv(const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
                                     sink_attn_bf16* k_cache, sink_attn_bf16* v_cache,
                                     int32_t num_pages, int32_t page_size,
                                     const int32_t* page_table, int32_t max_pages_per_seq,
                                     const int32_t* cu_seqlens, const int32_t* seq_lens,
                                     int32_t num_seqs, int32_t total_tokens, int32_t num_kv_heads,
                                     int32_t head_dim, sink_attn_stream_t stream);

/*
 * Ragged causal prefill whose keys are not the query rows themselves (contiguous K/V):
 * sequence s has queries cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (n_s rows) and keys
 * cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1 (m_s >= n_s rows); the queries are the last n_s
 * positions of the key range, so query row i of sequence s sits at position m_s - n_s + i
 * and sees keys j <= that position (and, with a window W > 0, position - j < W). With
 * cu_seqlens_k == cu_seqlens_q this is sink_attn_prefill. Uses: continuing a prefill from
 * a cached contiguous prefix, or cutting a long prefill into row chunks.
 *
 *   q, out     [total_q][num_q_heads][head_dim] bf16
 *   k, v       [total_k][num_kv_heads][head_dim] bf16
 *   cu_seqlens_q, cu_seqlens_k  [num_seqs + 1] int32, device
 *   max_seqlen_q, max_seqlen_k  host-side bounds of every n_s and every m_s
 *   lse        [total_q][num_q_heads] fp32 natural log, or NULL
 * A sequence with m_s < n_s, or key rows outside [0, total_k), is skipped and recorded in the
 * device error word (SINK_ATTN_DEVERR_SEQ_LEN / _CU_SEQLENS). Otherwise as sink_attn_prefill.
 */
sink_attn_status sink_attn_prefill_varlen(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                          const sink_attn_bf16* v, const float* sinks,
                                          const int32_t* cu_seqlens_q,
                                          const int32_t* cu_seqlens_k, int32_t num_seqs,
                                          int32_t total_q, int32_t total_k, int32_t max_seqlen_q,
                                          int32_t max_seqlen_k, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t window,
                                          float scale, sink_attn_bf16* out, float* lse,
                                          sink_attn_stream_t stream);

/*
 * The ragged causal prefill of sink_attn_prefill with its inputs in host memory and its
 * output returned to host memory: the copies and the kernels of one call overlap.
 *
 *   q_host, out_host  [total_tokens][num_q_heads][head_dim] bf16, host memory
 *   k_host, v_host    [total_tokens][num_kv_heads][head_dim] bf16, host memory
 *   sinks_host        [num_q_heads] fp32 host memory, or NULL (no sink)
 *   cu_seqlens_host   [num_seqs + 1] int32 host memory: sequence s is rows
 *                     cu[s] .. cu[s+1]-1; non-decreasing, cu[0] >= 0, cu[num_seqs] <=
 *                     total_tokens (checked here, before anything is issued)
 *   q_dev .. out_dev  device buffers of the same shapes (caller-owned, 16-byte aligned);
 *                     rows outside [cu[0], cu[num_seqs]) are neither copied nor written
 *   scratch           device memory of sink_attn_prefill_from_host_scratch_bytes(num_seqs,
 *                     num_q_heads, n_ranges) bytes, 16-byte aligned
 *   copy_in, copy_out streams for the host-to-device and device-to-host copies; NULL
 *                     puts that direction on `stream` (no overlap)
 *
 * The rows cu[0] .. cu[num_seqs]-1 are cut into n_ranges equal ranges, in order, across
 * sequence boundaries. Per range: its Q, K and V rows are copied in on copy_in;
 * sink_attn_prefill_varlen runs on `stream` with the range's rows as queries and each
 * range-sequence's rows from the sequence's first row as keys (earlier ranges copied those
 * in); its output rows are copied out on copy_out. Range g+1's input and range g-1's
 * output move while range g computes. The output equals that of sink_attn_prefill over
 * the whole batch up to rounding (a cut moves a sequence's q-tile boundaries).
 *
 * The call returns once everything is issued; it does not wait for the device. `stream`
 * is ordered after the last copy, so synchronising it makes out_host valid. The host
 * arrays must stay valid and unchanged until then, and should be page-locked (pinned)
 * for the copies to overlap. copy_in first waits for the work already on `stream` (the
 * device buffers may still be in use). Errors in the arguments are reported before
 * anything is issued; a CUDA error while issuing returns SINK_ATTN_ERR_CUDA and leaves
 * the outputs undefined.
 */
size_t sink_attn_prefill_from_host_scratch_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t n_ranges);
sink_attn_status sink_attn_prefill_from_host(
    const sink_attn_bf16* q_host, const sink_attn_bf16* k_host, const sink_attn_bf16* v_host,
    const float* sinks_host, const int32_t* cu_seqlens_host, int32_t num_seqs,
    int32_t total_tokens, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t window, float scale, sink_attn_bf16* out_host, sink_attn_bf16* q_dev,
    sink_attn_bf16* k_dev, sink_attn_bf16* v_dev, sink_attn_bf16* out_dev, void* scratch,
    size_t scratch_bytes, int32_t n_ranges, sink_attn_stream_t stream,
    sink_attn_stream_t copy_in, sink_attn_stream_t copy_out);

/*
 * Chunked prefill over the paged cache: appends the new rows' K/V (as
 * sink_attn_append_kv), then runs the ragged causal prefill of the new queries against
 * every cached key of their sequence. New query row i of sequence s sits at position
 * p = seq_lens[s] - n_s + i and sees cache positions j <= p (and p - j < W with a
 * window W > 0): the earlier chunks or prefix already in the cache plus the new rows.
 * With no earlier tokens (seq_lens[s] == n_s) this is sink_attn_prefill over the chunk.
 *
 *   q          [total_tokens][num_q_heads][head_dim] bf16 (new rows only)
 *   k_new, v_new, k_cache, v_cache, page_table, cu_seqlens, seq_lens: as
 *              sink_attn_append_kv
 *   max_q_len  host-side bound of every n_s; max_seq_len host-side bound of seq_lens
 *   sinks, window, scale: as sink_attn_prefill
 *   out        [total_tokens][num_q_heads][head_dim] bf16
 *   lse        [total_tokens][num_q_heads] fp32 (natural log), or NULL
 * Same support and error rules as sink_attn_prefill and sink_attn_append_kv.
 */
sink_attn_status sink_attn_prefill_paged(
    const sink_attn_bf16* q, const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
    sink_attn_bf16* k_cache, sink_attn_bf16* v_cache, int32_t num_pages, int32_t page_size,
    const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* cu_seqlens,
    const int32_t* seq_lens, int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
    int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    const float* sinks, int32_t window, float scale, sink_attn_bf16* out, float* lse,
    sink_attn_stream_t stream);

/*
 * Log-sum-exp outputs and the merge of attention states (cascade / shared-prefix
 * attention). This is the split-KV combination of "GPT-OSS am Day 0",
 * §Sink-Attention ¶2-¶3 made available to callers.
 *
 * The state of query row i of head h over a key set K is the pair
 *     lse = ln( e^{sink[h]} [only if the sink is counted] + sum_{j in K} e^{s_ij} )
 *     o   = sum_{j in K} e^{s_ij - lse} v_j
 * so a call over all visible keys returns exactly (out, ln Z) of the formula at the
 * top of this file (lse = m + ln Z there). An empty state (no key, no sink) is
 * (o = 0, lse = -inf); a state with only the sink is (o = 0, lse = sink[h]).
 * For two states over disjoint key sets A and B, the sink counted in at most one of
 * them, the state over A and B together is
 *     lse = ln(e^{lse_a} + e^{lse_b}),   o = e^{lse_a - lse} o_a + e^{lse_b - lse} o_b.
 * Example: decode every request against a shared prefix (its pages, with the sinks)
 * and against its own suffix (sinks NULL), then merge the two states.
 *
 * sink_attn_prefill_lse and sink_attn_decode_lse take the arguments of
 * sink_attn_prefill / sink_attn_decode plus
 *   lse   fp32 [total_tokens][num_q_heads] (prefill) or [batch][num_q_heads] (decode),
 *         natural logarithm, 4-byte aligned; rows of tokens that belong to no
 *         sequence are not written.
 * and return the same `out`.
 */
sink_attn_status sink_attn_prefill_lse(const sink_attn_bf16* q, const sink_attn_bf16* k,
                                       const sink_attn_bf16* v, const float* sinks,
                                       const int32_t* cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_seqlen,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t window, float scale,
                                       sink_attn_bf16* out, float* lse,
                                       sink_attn_stream_t stream);

sink_attn_status sink_attn_decode_lse(const sink_attn_bf16* q, const sink_attn_bf16* k_cache,
                                      const sink_attn_bf16* v_cache, int32_t num_pages,
                                      int32_t page_size, const int32_t* page_table,
                                      int32_t max_pages_per_seq, const int32_t* seq_lens,
                                      int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, const float* sinks,
                                      int32_t window, float scale, int32_t kv_chunk,
                                      void* workspace, size_t workspace_bytes,
                                      sink_attn_bf16* out, float* lse,
                                      sink_attn_stream_t stream);

/*
 * Merge two attention states row by row (formula above).
 *   o_a, o_b   [rows][num_heads][head_dim] bf16 (for example the `out` of two calls)
 *   lse_a, lse_b [rows][num_heads] fp32, natural logarithm (may be -inf)
 *   o_out      [rows][num_heads][head_dim] bf16; must not overlap the inputs
 *   lse_out    [rows][num_heads] fp32, or NULL when not wanted
 * The arithmetic is fp32; the merged o is rounded to bf16 once.
 * Supported: head_dim in {64, 128}; rows * num_heads < 2^31.
 */
sink_attn_status sink_attn_merge_states(const sink_attn_bf16* o_a, const float* lse_a,
                                        const sink_attn_bf16* o_b, const float* lse_b,
                                        int32_t rows, int32_t num_heads, int32_t head_dim,
                                        sink_attn_bf16* o_out, float* lse_out,
                                        sink_attn_stream_t stream);

/*
 * FP8 KV cache. The pages quantise to 8-bit floating point with scale factors
 * ("Qwen hosten op Blackwell", §Kwantisering); this cache format applies that to K and V:
 *   k_codes, v_codes  [num_pages][num_kv_heads][page_size][head_dim] uint8, e4m3 codes
 *                     (OCP E4M3: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *                     subnormals, largest finite 448, S.1111.111 is NaN)
 *   k_scale, v_scale  [num_pages][num_kv_heads][page_size] fp32, one scale per row
 * The value of element d of a cached token row is e4m3(code[d]) * scale. Per token the
 * cache holds 2 * num_kv_heads * (head_dim + 4) bytes instead of 4 * num_kv_heads *
 * head_dim. All buffers are caller-owned device memory, 16-byte aligned.
 *
 * Quantisation of a bf16 row x (IEEE fp32 arithmetic, round to nearest even):
 *   amax = max |x_d|;  scale = amax / 448;  code_d = e4m3_satfinite(x_d * (448 / amax))
 * so the row's largest element becomes +-448; a zero row has scale 0 and zero codes.
 * Range: the decode keeps V-row scales below 2^8 (|v| below 114688) and any finite K.
 */

/* Quantise `rows` contiguous bf16 rows x [rows][head_dim] into codes [rows][head_dim]
 * and scales [rows] (for example a whole bf16 cache: rows = num_pages * num_kv_heads *
 * page_size). head_dim in {64, 128}. */
sink_attn_status sink_attn_quantize_fp8(const sink_attn_bf16* x, int64_t rows, int32_t head_dim,
                                        uint8_t* codes, float* scales, sink_attn_stream_t stream);

/* sink_attn_append_kv for the FP8 cache: each new K and V row is quantised into its slot
 * (codes and scale); same arguments, placement and error rules. */
sink_attn_status sink_attn_append_kv_fp8(const sink_attn_bf16* k_new, const sink_attn_bf16* v_new,
                                         uint8_t* k_codes, uint8_t* v_codes, float* k_scale,
                                         float* v_scale, int32_t num_pages, int32_t page_size,
                                         const int32_t* page_table, int32_t max_pages_per_seq,
                                         const int32_t* cu_seqlens, const int32_t* seq_lens,
                                         int32_t num_seqs, int32_t total_tokens,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         sink_attn_stream_t stream);

/* sink_attn_decode over the FP8 cache: the arguments of sink_attn_decode with the bf16
 * pages replaced by codes and row scales, plus `lse` ([batch][num_q_heads] fp32 natural
 * log, or NULL). The workspace is sized by sink_attn_decode_workspace_bytes as for bf16.
 * Q stays bf16; scores and the softmax are fp32 as in the bf16 decode. */
sink_attn_status sink_attn_decode_fp8(const sink_attn_bf16* q, const uint8_t* k_codes,
                                      const uint8_t* v_codes, const float* k_scale,
                                      const float* v_scale, int32_t num_pages, int32_t page_size,
                                      const int32_t* page_table, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      const float* sinks, int32_t window, float scale,
                                      int32_t kv_chunk, void* workspace, size_t workspace_bytes,
                                      sink_attn_bf16* out, float* lse, sink_attn_stream_t stream);

/* Scratch bytes sink_attn_decode needs for these sizes (0 when every sequence
 * fits one chunk). Pure host arithmetic; returns 0 for invalid sizes. */
size_t sink_attn_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                        int32_t max_seq_len, int32_t kv_chunk);

/* Static, human-readable name of a status code. */
const char* sink_attn_status_string(sink_attn_status status);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device (bits SINK_ATTN_DEVERR_*) in *bits_out (may be NULL).
 * Returns SINK_ATTN_ERR_DEVICE if any bit was set, SINK_ATTN_ERR_CUDA if the
 * synchronisation failed, else SINK_ATTN_OK. */
sink_attn_status sink_attn_read_device_error(sink_attn_stream_t stream, uint32_t* bits_out);

/* Number of streaming multiprocessors the library sizes persistent grids for
 * on the current device (0 if no device is visible). Host query only. */
int32_t sink_attn_num_sms(void);

/*
 * Test switch for the decode's failure path; the pages have no counterpart. With
 * enable != 0, every later decode launch (sink_attn_decode, _decode_lse, _decode_fp8,
 * _decode_static_workspace) never copies the first page of (chunk 0, kv head 0,
 * sequence 0): the consumer warps' wait for it runs out after wait_limit_ns, the CTA
 * sets SINK_ATTN_DEVERR_WAIT_TIMEOUT in the device error word, lets its copies in
 * flight land (those waits keep their own 1 s limit), and returns without writing that
 * sequence's partial results; every other CTA runs normally. Nothing traps and nothing
 * waits without a limit. enable == 0 restores the normal launches (and the 1 s limit).
 * The switch is process-wide, not per stream or thread: it exists for tests only.
 */
void sink_attn_debug_decode_withhold_page(int32_t enable, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SINK_ATTN_H */
