// decode_split.cu — paged split-KV decode with a per-head sink logit, and the
// log-sum-exp merge of the chunks.
//
// One CTA per (chunk, kv head, sequence): a producer warp streams the chunk's
// (page, kv head) blocks of K and V — each a contiguous page_size x head_dim tile of
// the HND cache ("Qwen hosten op Blackwell", §Inzet op GB200 NVL72) — with TMA into
// a ring of 128-byte-swizzled shared-memory stages; four consumer warps (one
// warpgroup serving the whole GQA query group of that kv head) take the pages in
// turn. Decode is memory-bound ("Qwen hosten op Blackwell", §Decoders), so the
// small per-page contractions (16 tokens x head_dim x group) run on warp-level
// bf16 MMAs purely to keep the FP32 pipes from becoming the limit.
//
// Online softmax in the exp2 domain; the running maximum of every query head
// starts from its sink value only in the chunk that begins the visible range, and
// from -inf in every other chunk ("GPT-OSS am Day 0", §Sink-Attention ¶3). Chunks
// emit (normalised partial output, log2-sum-exp); a merge kernel combines them
// with warp-shuffle reductions. A sequence that fits one chunk is finished by the
// split kernel directly and the merge skips it.
//
// FP8 cache (template flag F8): K and V pages hold e4m3 codes, with one fp32 scale
// per (token, kv head) row in separate arrays; a token's values are code * scale
// (the 8-bit floating-point direction of "Qwen hosten op Blackwell", §Kwantisering).
// The pages move with TMA as bytes (half the bf16 traffic) and the row scales with
// bulk copies; consumers convert codes to f16 in registers (exact for every e4m3
// value) and run f16 warp MMAs:
//   S = K Q^T: ldmatrix on byte pairs gives each lane k-consecutive codes 4t..4t+3
//     of a 16-wide slice, so the A fragment's k order is permuted within the slice;
//     Q's B fragment is built with the same permutation (the dot product is
//     order-free). Q is scaled by a power of two into f16 range; the K row scale
//     and that power multiply S in fp32.
//   O^T += V^T P: ldmatrix.trans on byte pairs gives two head_dim rows per register;
//     one byte permute splits them into an even-row and an odd-row A fragment, so a
//     32-row slice of head_dim is two MMAs whose output rows interleave. The V row
//     scale (times 2^8, undone at the end) multiplies P before its f16 rounding.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kPage = 16;          // tokens per page
constexpr int kConsumerWarps = 4;  // one warpgroup
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr float kPvScale = 256.f;  // FP8 path: P carries v_scale * 2^8 into the f16 MMA

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const float* sinks;
  const float* k_scale;  // FP8 cache: [pages, Hkv, 16] fp32 row scales
  const float* v_scale;
  __nv_bfloat16* out;
  float* lse_out;  // [B, Hq] natural log, or null
  float* o_part;
  float* lse_part;
  unsigned* err;
  int num_pages, max_pages, batch, max_seq_len, Hq, Hkv, G, window, chunk, cmax;
  float scale_log2;
  uint64_t timeout_ns;  // pipeline waits
  uint64_t drain_ns;    // teardown waits for copies in flight
  int withhold;         // test switch (see DecodeLaunch::withhold_first_page)
};

// Sequence length as used by both kernels: out-of-contract values are recorded
// and clamped so the grid and the page table are never overrun.
__device__ __forceinline__ int checked_len(const DecodeParams& p, int b, bool report) {
  int L = p.seq_lens[b];
  int bound = p.max_seq_len;
  if (p.max_pages * kPage < bound) bound = p.max_pages * kPage;
  if (L < 0 || L > bound) {
    if (report) atomicOr(p.err, kErrSeqLen);
    L = L < 0 ? 0 : bound;
  }
  return L;
}

__device__ __forceinline__ void visible_range(const DecodeParams& p, int L, int& lo, int& nch) {
  lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  int nvis = L - lo;
  nch = nvis > 0 ? (nvis + p.chunk - 1) / p.chunk : 1;
}

// ST = pages in flight per CTA (ring depth); launch_split picks it.
template <int D, int NT, bool F8, int ST>
struct DecodeSmem {
  static constexpr int kStages = ST;
  static constexpr int kRowBytes = F8 ? D : 2 * D;      // one token row of one head
  static constexpr int kBoxes = F8 ? 1 : D / 64;        // TMA boxes per page
  static constexpr int kPageBytes = kPage * kRowBytes;  // one (page, head) block
  static constexpr int kStageBytes = 2 * kPageBytes;    // K + V
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kScaleBytes = F8 ? 2 * kPage * 4 : 0;  // K and V row scales
  static constexpr int kScaleOffset = kRingBytes;
  static constexpr int kBarOffset = kScaleOffset + kStages * kScaleBytes;  // full[], empty[]
  static constexpr int kFlagOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kBytes = kFlagOffset + 16 + 1024;  // + alignment slack
  static constexpr int kTxBytes = kStageBytes + kScaleBytes;
  // Consumer warp w takes pages w, w + 4, ...; page i uses stage i % kStages. With a ring
  // depth that is a multiple of the consumer warps, the next use of a stage goes to the warp
  // that consumed its previous page, so no full-barrier wait is ever two phases ahead (where
  // the parity would match an already completed phase and the wait would pass early).
  static constexpr int kGroups = (NT == 2 && !F8) ? 2 : kConsumerWarps;  // page owners per round
  static_assert(kStages % kGroups == 0, "ring depth must be a multiple of the consumer groups");
};

// Shared-memory byte address of 16-byte chunk `c` of token row `r` (0..15) in a page
// block written by TMA: bf16 rows are D/64 boxes of 128 bytes (128-byte swizzle); FP8
// rows are one box of D bytes (64-byte swizzle at D = 64, 128-byte at D = 128).
template <int D, bool F8>
__device__ __forceinline__ uint32_t page_chunk_addr(uint32_t base, int r, int c) {
  if constexpr (F8 && D == 64) {
    return base + r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
  } else if constexpr (F8) {
    return base + r * 128 + ((c ^ (r & 7)) << 4);
  } else {
    const int box = c >> 3;
    const int cc = c & 7;
    return base + box * (kPage * 128) + r * 128 + ((cc ^ (r & 7)) << 4);
  }
}

// The split kernel's body; the __global__ entry points below differ only in their
// launch bounds. tm_k and tm_v are the kernel's __grid_constant__ parameters.
template <int D, int NT, bool F8, int ST>
__device__ __forceinline__ void decode_split_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                                  const DecodeParams& p) {
  using S = DecodeSmem<D, NT, F8, ST>;
  constexpr int kStages = S::kStages;
  constexpr bool kSplitTiles = (NT == 2) && !F8;  // each consumer warp serves one head tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_full = sbase + S::kBarOffset;
  const uint32_t bar_empty = bar_full + kStages * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kFlagOffset);

  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The merge kernel (launched as a programmatic dependent) may be scheduled once every
  // CTA of this grid has started; it waits for this grid's completion before reading.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int L = checked_len(p, b, c == 0 && g == 0 && threadIdx.x == 0);
  int vis_lo, nch;
  visible_range(p, L, vis_lo, nch);
  if (c >= nch) return;  // uniform for the whole CTA
  const int t_lo = vis_lo + c * p.chunk;
  const int t_hi = min(t_lo + p.chunk, L);
  const int p_first = t_lo / kPage;
  const int npg = (t_hi > t_lo) ? (t_hi - 1) / kPage - p_first + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kSplitTiles ? 2 : 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == kConsumerWarps) {
    // ---------------- producer: the whole warp walks the pages, one lane issues ----------------
    // Page-table entries are read 32 at a time (one per lane), one block ahead, so no
    // TMA issue waits on a dependent global load; a page's id is taken by a shuffle.
    if (npg > 0) {
      if (elect_one()) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      const int32_t* pt = p.page_table + (size_t)b * p.max_pages + p_first;
      int cur = lane < npg ? pt[lane] : -1;
      int nxt = 32 + lane < npg ? pt[32 + lane] : -1;
      // Test switch: page 0 of (chunk 0, kv head 0, sequence 0) is never copied (the loop
      // starts at page 1), so the consumers' bounded wait for it runs out and the CTA
      // aborts through its normal path.
      const int first = (p.withhold && c == 0 && g == 0 && b == 0) ? 1 : 0;
      int issued = first;
      for (int i = first; i < npg; ++i) {
        if (i > 0 && (i & 31) == 0) {
          cur = nxt;
          nxt = i + 32 + lane < npg ? pt[i + 32 + lane] : -1;
        }
        const int pid = __shfl_sync(0xffffffffu, cur, i & 31);
        const int st = i % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * st, ((i / kStages) & 1) ^ 1, wc)))
          break;
        if (elect_one()) {
          const uint32_t full = bar_full + 8 * st;
          if (pid < 0 || pid >= p.num_pages) {
            atomicOr(p.err, kErrPageId);
            mbar_arrive(full);  // release the consumer; the stage keeps stale data
          } else {
            mbar_arrive_expect_tx(full, S::kTxBytes);
            const uint32_t kdst = sbase + st * S::kStageBytes;
            const uint32_t vdst = kdst + S::kPageBytes;
            const int row = (pid * p.Hkv + g) * kPage;
#pragma unroll
            for (int bx = 0; bx < S::kBoxes; ++bx) {
              tma_load_2d(kdst + bx * kPage * 128, &tm_k, full, bx * 64, row);
              tma_load_2d(vdst + bx * kPage * 128, &tm_v, full, bx * 64, row);
            }
            if constexpr (F8) {
              const uint32_t sdst = sbase + S::kScaleOffset + st * S::kScaleBytes;
              bulk_load(sdst, p.k_scale + row, kPage * 4, full);
              bulk_load(sdst + kPage * 4, p.v_scale + row, kPage * 4, full);
            }
          }
        }
        __syncwarp();
        issued = i + 1;
      }
      // Let every copy still in flight land before the CTA can exit.
      if (lane == 0) {
        for (int i = max(first, issued - kStages); i < issued; ++i)  // pages copied
          mbar_drain(bar_full + 8 * (i % kStages), (i / kStages) & 1, p.drain_ns);
      }
    }
    return;
  }

  // ---------------- consumers: warp w takes pages w, w+4, w+8, ... ----------------
  const int G = p.G;
  const int head0 = g * G;
  // Two head tiles of a bf16 cache (a group of 16): warps 0-1 serve tile 0 and warps 2-3
  // tile 1, each pair taking the even / odd pages, so a warp holds the Q fragments and
  // running outputs of one tile only (92 registers instead of 128 with spills: four CTAs
  // per SM instead of three). Otherwise every warp serves all tiles of its pages.
  constexpr int NTW = kSplitTiles ? 1 : NT;  // head tiles per warp
  const int tile0 = kSplitTiles ? (warp >> 1) : 0;
  const int pfirst = kSplitTiles ? (warp & 1) : warp;
  constexpr int pstep = kSplitTiles ? 2 : kConsumerWarps;
  // Q of the group as B fragments of S = K * Q^T (k = head_dim, n = query head).
  // bf16: lane (g, t) holds head_dim pairs 2t, 2t+1 and 2t+8, 2t+9 of each 16-wide slice.
  // FP8: f16, pairs 4t, 4t+1 and 4t+2, 4t+3 (the permuted k order of the K fragments),
  // scaled by 2^-qexp so that the group's largest |q| is below 2^15.
  uint32_t qf[NTW][D / 16][2];
  float qmul = 1.f;  // FP8: 2^qexp, applied to S in fp32
  if constexpr (F8) {
    auto q_quad = [&](int nt, int kk) {  // head_dim 16kk + 4t .. +3 of head nt*8 + g
      const int hl = (tile0 + nt) * 8 + (lane >> 2);
      if (hl >= G) return make_uint2(0u, 0u);
      const __nv_bfloat16* qrow = p.q + ((size_t)b * p.Hq + head0 + hl) * D;
      return *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * (lane & 3));
    };
    float qmax = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint2 raw = q_quad(nt, kk);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(hi.x), fabsf(hi.y))));
      }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
    const int e = (int)((__float_as_uint(qmax) >> 23) & 0xFF) - 127;  // floor(log2 qmax)
    const int qexp = e >= 15 ? min(e - 14, 100) : 0;
    qmul = __int_as_float((127 + qexp) << 23);
    const float down = __int_as_float((127 - qexp) << 23);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint2 raw = q_quad(nt, kk);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        qf[nt][kk][0] = pack_f16x2(lo.x * down, lo.y * down);
        qf[nt][kk][1] = pack_f16x2(hi.x * down, hi.y * down);
      }
  } else {
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      const int hl = (tile0 + nt) * 8 + (lane >> 2);
      const bool hv = hl < G;
      const uint32_t* qrow =
          reinterpret_cast<const uint32_t*>(p.q + ((size_t)b * p.Hq + head0 + (hv ? hl : 0)) * D);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qf[nt][kk][0] = hv ? qrow[(kk * 16 + 2 * (lane & 3)) >> 1] : 0u;
        qf[nt][kk][1] = hv ? qrow[(kk * 16 + 8 + 2 * (lane & 3)) >> 1] : 0u;
      }
    }
  }
  float m[NTW][2], l[NTW][2];
  float o[NTW][D / 16][4];
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
  }
  const float sl = p.scale_log2 * qmul;
  bool aborted = false;

  for (int i = pfirst; i < npg; i += pstep) {
    const int st = i % kStages;
    bool ok = mbar_wait(bar_full + 8 * st, (i / kStages) & 1, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      aborted = true;
      break;
    }
    const uint32_t kbase = sbase + st * S::kStageBytes;
    const uint32_t vbase = kbase + S::kPageBytes;
    const int tok0 = (p_first + i) * kPage;
    const bool partial = tok0 < t_lo || tok0 + kPage > t_hi;
    if (partial) {
      // Positions outside [t_lo, t_hi) may hold anything (even NaN): zero their
      // value rows so that p = 0 cannot meet a non-finite v in the MMA.
      constexpr int kRowChunks = S::kRowBytes / 16;
      for (int idx = lane; idx < kPage * kRowChunks; idx += 32) {
        const int r = idx / kRowChunks, cch = idx % kRowChunks;
        const int t = tok0 + r;
        if (t < t_lo || t >= t_hi) {
          const uint32_t a = page_chunk_addr<D, F8>(vbase, r, cch);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
      }
      __syncwarp();
    }
    // S[16 tokens x 8 heads] per head tile.
    float s[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const int mat = lane >> 3, rr = lane & 7;
    if constexpr (F8) {
#pragma unroll
      for (int kc = 0; kc < D / 32; ++kc) {
        // matrices: tokens 0-7 / 8-15 of 16-byte chunk 2kc, then of chunk 2kc + 1
        uint32_t r[4];
        ldsm_x4(page_chunk_addr<D, true>(kbase, rr + ((mat & 1) << 3), 2 * kc + (mat >> 1)), r);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t a[4];
          e4m3x4_to_f16x2x2(r[2 * hf], a[0], a[2]);      // token g: codes 4t, 4t+1 | 4t+2, 4t+3
          e4m3x4_to_f16x2x2(r[2 * hf + 1], a[1], a[3]);  // token g+8
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt)
            mma_16816_f16(s[nt], a, qf[nt][2 * kc + hf][0], qf[nt][2 * kc + hf][1]);
        }
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(page_chunk_addr<D, false>(kbase, rr + ((mat & 1) << 3), 2 * kk + (mat >> 1)), a);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) mma_16816(s[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
      }
    }
    const int ta = tok0 + (lane >> 2), tb = ta + 8;
    const bool va = ta >= t_lo && ta < t_hi, vb = tb >= t_lo && tb < t_hi;
    // score factors per token row (FP8: times the K row scale) and P factors (FP8: the
    // V row scale times 2^8; 0 for positions outside the range, whose scales may be junk)
    float fa = sl, fb = sl, pa = 1.f, pb_ = 1.f;
    if constexpr (F8) {
      const float* sc = reinterpret_cast<const float*>(smem + S::kScaleOffset + st * S::kScaleBytes);
      const int ra = lane >> 2;
      fa = sl * sc[ra];
      fb = sl * sc[ra + 8];
      pa = va ? sc[kPage + ra] * kPvScale : 0.f;
      pb_ = vb ? sc[kPage + ra + 8] * kPvScale : 0.f;
    }
    uint32_t pb[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      const float x0 = va ? s[nt][0] * fa : -INFINITY;  // token a, head A
      const float x1 = va ? s[nt][1] * fa : -INFINITY;  // token a, head B
      const float x2 = vb ? s[nt][2] * fb : -INFINITY;  // token b, head A
      const float x3 = vb ? s[nt][3] * fb : -INFINITY;  // token b, head B
      float mxa = fmaxf(x0, x2), mxb = fmaxf(x1, x3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
      }
      const float mna = fmaxf(m[nt][0], mxa), mnb = fmaxf(m[nt][1], mxb);
      const float mua = mna == -INFINITY ? 0.f : mna, mub = mnb == -INFINITY ? 0.f : mnb;
      const float aa = ex2(m[nt][0] - mua), ab = ex2(m[nt][1] - mub);
      const float p0 = ex2(x0 - mua), p2 = ex2(x2 - mua);
      const float p1 = ex2(x1 - mub), p3 = ex2(x3 - mub);
      l[nt][0] = l[nt][0] * aa + (p0 + p2);
      l[nt][1] = l[nt][1] * ab + (p1 + p3);
      m[nt][0] = mna;
      m[nt][1] = mnb;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[nt][mt][0] *= aa;
        o[nt][mt][1] *= ab;
        o[nt][mt][2] *= aa;
        o[nt][mt][3] *= ab;
      }
      if constexpr (F8) {
        pb[nt][0] = movmatrix_trans(pack_f16x2(p0 * pa, p1 * pa));
        pb[nt][1] = movmatrix_trans(pack_f16x2(p2 * pb_, p3 * pb_));
      } else {
        pb[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
        pb[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
      }
    }
    // O^T[head_dim x heads] += V^T[head_dim x 16 tokens] * P[16 tokens x heads]
    if constexpr (F8) {
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        // matrices: tokens 0-7 of chunks 2j, 2j+1, then tokens 8-15 of the same chunks;
        // lane (g, t) receives, per matrix, the codes of head_dim rows 2g, 2g+1 of the
        // chunk for tokens 2t, 2t+1 (bytes: [2t][2g], [2t][2g+1], [2t+1][2g], [2t+1][2g+1])
        uint32_t r[4];
        ldsm_x4_trans(page_chunk_addr<D, true>(vbase, rr + ((mat >> 1) << 3), 2 * j + (mat & 1)), r);
        uint32_t ae[4], ao[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t sp = prmt(r[x], 0u, 0x3120u);  // {even row: t0 t1, odd row: t0 t1}
          e4m3x4_to_f16x2x2(sp, ae[x], ao[x]);
        }
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          mma_16816_f16(o[nt][2 * j], ae, pb[nt][0], pb[nt][1]);
          mma_16816_f16(o[nt][2 * j + 1], ao, pb[nt][0], pb[nt][1]);
        }
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(page_chunk_addr<D, false>(vbase, rr + ((mat >> 1) << 3), 2 * mt + (mat & 1)), a);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) mma_16816(o[nt][mt], a, pb[nt][0], pb[nt][1]);
      }
    }
    if (partial) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);
  }

  // ---------------- combine the four warps (and the sink) ----------------
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");  // ring is free now
  if (*abort_flag) aborted = true;
  constexpr int GP = NTW * 8;  // heads held per warp (padded)
  static_assert((kConsumerWarps * GP * (2 + D) + 16 * kConsumerWarps) * 4 <= S::kRingBytes,
                "the combine scratch must fit in the ring it reuses");
  float* cm = reinterpret_cast<float*>(smem);  // [4][GP]
  float* cl = cm + kConsumerWarps * GP;        // [4][GP]
  float* co = cl + kConsumerWarps * GP;        // [4][GP][D]
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
      l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
    }
    const int ha = nt * 8 + 2 * (lane & 3);
    if (lane < 4) {
      cm[warp * GP + ha] = m[nt][0];
      cm[warp * GP + ha + 1] = m[nt][1];
      cl[warp * GP + ha] = l[nt][0];
      cl[warp * GP + ha + 1] = l[nt][1];
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      // output rows of tile mt held by this lane: bf16 d, d + 8; FP8 (even/odd interleave of
      // a 32-row slice) d = 32*(mt/2) + 2g + mt%2 and d + 16, carrying the factor 2^8
      const int gq = lane >> 2;
      const int d = F8 ? 32 * (mt >> 1) + 2 * gq + (mt & 1) : mt * 16 + gq;
      const int d2 = F8 ? d + 16 : d + 8;
      const float f = F8 ? 1.f / kPvScale : 1.f;
      co[(warp * GP + ha) * D + d] = o[nt][mt][0] * f;
      co[(warp * GP + ha + 1) * D + d] = o[nt][mt][1] * f;
      co[(warp * GP + ha) * D + d2] = o[nt][mt][2] * f;
      co[(warp * GP + ha + 1) * D + d2] = o[nt][mt][3] * f;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
  if (aborted) return;

  // Per head: each holding warp's weight 2^(m_w - M) / d (the sink counted once, in the
  // first chunk of the visible range) and the chunk's log-sum-exp, once per head instead of
  // once per output element.
  constexpr int NW = kSplitTiles ? 2 : kConsumerWarps;  // warps holding one head
  float* cwt = co + kConsumerWarps * GP * D;            // [G][NW]
  if (threadIdx.x < G) {
    const int hl = threadIdx.x;
    const int h = head0 + hl;
    const int w0 = kSplitTiles ? 2 * (hl >> 3) : 0;
    const int hh = kSplitTiles ? (hl & 7) : hl;
    const float sink_l2 = (c == 0 && p.sinks != nullptr) ? p.sinks[h] * kLog2e : -INFINITY;
    float M = sink_l2;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[(w0 + w) * GP + hh]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float lsum = ex2(sink_l2 - Mu);
    float f[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      f[w] = ex2(cm[(w0 + w) * GP + hh] - Mu);
      lsum += cl[(w0 + w) * GP + hh] * f[w];
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) cwt[hl * NW + w] = f[w] * inv;
    const size_t bh = (size_t)b * p.Hq + h;
    if (nch == 1) {
      if (p.lse_out) p.lse_out[bh] = lsum > 0.f ? (Mu + log2f(lsum)) * kLn2 : -INFINITY;
    } else {
      p.lse_part[bh * p.cmax + c] = lsum > 0.f ? Mu + __log2f(lsum) : -INFINITY;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
  // The weighted sums, four consecutive head_dim elements per thread.
  for (int idx = threadIdx.x; idx < G * D / 4; idx += kConsumerWarps * 32) {
    const int hl = idx / (D / 4), d = 4 * (idx % (D / 4));
    const int w0 = kSplitTiles ? 2 * (hl >> 3) : 0;
    const int hh = kSplitTiles ? (hl & 7) : hl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = cwt[hl * NW + w];
      const float4 x = *reinterpret_cast<const float4*>(co + ((w0 + w) * GP + hh) * D + d);
      acc.x += x.x * f;
      acc.y += x.y * f;
      acc.z += x.z * f;
      acc.w += x.w * f;
    }
    const size_t bh = (size_t)b * p.Hq + head0 + hl;
    if (nch == 1) {
      uint2 v;
      v.x = pack_bf16x2(acc.x, acc.y);
      v.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.out + bh * D + d) = v;
    } else {
      *reinterpret_cast<float4*>(p.o_part + (bh * p.cmax + c) * D + d) = acc;
    }
  }
}

template <int D, int NT, bool F8, int ST>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  decode_split_body<D, NT, F8, ST>(tm_k, tm_v, p);
}

// Two head tiles at head_dim 128 (a group of 16 query heads): registers, not shared memory,
// bound the resident CTAs, and the latency-bound consumers gain from more of them. FP8
// cache (every warp serves both tiles): capped for three CTAs per SM. bf16 cache (one tile
// per warp, 92 registers): four CTAs per SM, Qwen3-235B-style decode 0.1471 -> 0.1409 ms.
template <int D, int NT, bool F8, int ST>
__global__ void __launch_bounds__(kDecodeThreads, F8 ? 3 : 4)
    decode_split_kernel_3(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  decode_split_body<D, NT, F8, ST>(tm_k, tm_v, p);
}

// FP8 cache at head_dim 64 with one head tile: capped for seven CTAs per SM (56 registers),
// the residency its shared memory allows; left to itself the compiler takes 60, which
// leaves room for six.
template <int D, int NT, bool F8, int ST>
__global__ void __launch_bounds__(kDecodeThreads, 7)
    decode_split_kernel_7(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  decode_split_body<D, NT, F8, ST>(tm_k, tm_v, p);
}

// One warp per (sequence, query head): out = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M).
// Launched as a programmatic dependent of the split kernel; chunk rows are read eight at a
// time so their loads overlap instead of forming a dependent chain.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the split grid's results are visible
  constexpr int V = D / 32;  // consecutive head_dim elements per lane
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.batch * p.Hq) return;
  const int b = wid / p.Hq;
  const int L = checked_len(p, b, false);
  int vis_lo, nch;
  visible_range(p, L, vis_lo, nch);
  if (nch <= 1) return;  // finished by the split kernel
  const float* lse = p.lse_part + (size_t)wid * p.cmax;
  const float* op = p.o_part + (size_t)wid * p.cmax * D + lane * V;
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, lse[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Mu = M == -INFINITY ? 0.f : M;
  float W = 0.f;  // the same in every lane: every lane sums the same weights in order
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 8) {
    float x[8][V], w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + k;
      const bool valid = c < nch;
      w[k] = valid ? ex2(lse[c] - Mu) : 0.f;
      if constexpr (V == 2) {
        const float2 v2 = valid ? *reinterpret_cast<const float2*>(op + (size_t)c * D) : make_float2(0.f, 0.f);
        x[k][0] = v2.x;
        x[k][1] = v2.y;
      } else {
        const float4 v4 = valid ? *reinterpret_cast<const float4*>(op + (size_t)c * D)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        x[k][0] = v4.x;
        x[k][1] = v4.y;
        x[k][2] = v4.z;
        x[k][3] = v4.w;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      W += w[k];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += w[k] * x[k][e];
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  if (lane == 0 && p.lse_out) p.lse_out[wid] = W > 0.f ? (Mu + log2f(W)) * kLn2 : -INFINITY;
  __nv_bfloat16* dst = p.out + (size_t)wid * D + lane * V;
#pragma unroll
  for (int e = 0; e < V; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

template <int D, int NT, bool F8, int ST>
cudaError_t launch_split_ring(const DecodeLaunch& a, const DecodeParams& p, cudaStream_t stream) {
  using S = DecodeSmem<D, NT, F8, ST>;
  auto kern = []() {
    if constexpr (NT == 2 && D == 128) return decode_split_kernel_3<D, NT, F8, ST>;
    else if constexpr (F8 && NT == 1 && D == 64) return decode_split_kernel_7<D, NT, F8, ST>;
    else return decode_split_kernel<D, NT, F8, ST>;
  }();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.cmax, a.num_kv_heads, a.batch);
  kern<<<grid, kDecodeThreads, S::kBytes, stream>>>(a.tm_k, a.tm_v, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.cmax <= 1) return e;
  const int warps = a.batch * a.num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
}

// Ring depth: FP8 12 pages (8 leaves no room for the combine scratch of two head tiles).
// bf16: 8, except when no CTA reads more than 9 pages (a window of at most 128 tokens,
// which may start inside a page): there every page fits a 4-page ring twice over, and the
// smaller ring lets more CTAs stay resident, so a grid of short ranges runs in fewer
// waves (long-context decode with a 128-token window: 17.2 -> 14.4 us). bf16 with two head
// tiles: 6 pages (4, 6 and 8 measured within 1% of each other; each warp pair owns every
// other page, so the depth must be even).
template <int D, int NT, bool F8>
cudaError_t launch_split(const DecodeLaunch& a, const DecodeParams& p, cudaStream_t stream) {
  if constexpr (F8) {
    return launch_split_ring<D, NT, F8, 12>(a, p, stream);
  } else {
    if constexpr (NT == 1) {
      const int vis = p.window > 0 ? min(p.window, p.max_seq_len) : p.max_seq_len;
      const int pages = (min(vis, p.chunk) + kPage - 1) / kPage + 1;
      if (pages <= 9) return launch_split_ring<D, NT, F8, 4>(a, p, stream);
    }
    if constexpr (NT == 2) return launch_split_ring<D, NT, F8, 6>(a, p, stream);
    else return launch_split_ring<D, NT, F8, 8>(a, p, stream);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream) {
  DecodeParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.sinks = a.sinks;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse_out = a.lse;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.err = a.err;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  p.batch = a.batch;
  p.max_seq_len = a.max_seq_len;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.G = a.num_q_heads / a.num_kv_heads;
  p.window = a.window;
  p.chunk = a.kv_chunk;
  p.cmax = a.cmax;
  p.scale_log2 = a.scale * kLog2e;
  p.timeout_ns = a.timeout_ns;
  p.drain_ns = a.drain_ns;
  p.withhold = a.withhold_first_page;
  const bool two_tiles = p.G > 8;
  if (a.fp8) {
    if (a.head_dim == 64)
      return two_tiles ? launch_split<64, 2, true>(a, p, stream) : launch_split<64, 1, true>(a, p, stream);
    return two_tiles ? launch_split<128, 2, true>(a, p, stream) : launch_split<128, 1, true>(a, p, stream);
  }
  if (a.head_dim == 64)
    return two_tiles ? launch_split<64, 2, false>(a, p, stream) : launch_split<64, 1, false>(a, p, stream);
  return two_tiles ? launch_split<128, 2, false>(a, p, stream) : launch_split<128, 1, false>(a, p, stream);
}

}  // namespace sa
