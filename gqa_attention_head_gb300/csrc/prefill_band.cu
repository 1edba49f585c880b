// prefill_band.cu — sliding-window prefill for short windows (1..128 keys) at head_dim 64,
// when each kv head serves a multiple of 8 query heads (the gpt-oss shape, 64 query / 8 kv
// heads, with a 128-token window). The sink softmax is that of "GPT-OSS am Day 0",
// §Sink-Attention; the pages do not describe windows, whose convention here is W keys, the
// query's own included.
//
// Work unit: 32 consecutive queries of one sequence, one kv head and 8 of its query heads.
// The 128 MMA rows of a head tile are 8 query heads x 16 queries, row r = 8 * query + head,
// exactly what one TMA box {64 dims, 8 heads, 16 tokens} of the [tokens][heads][dims] layout
// delivers; head tile t holds queries q0 + 16 t .. q0 + 16 t + 15. With a window of at most 128
// keys every row of the unit sees only keys in the span [q0 - 128, q0 + 32) of its sequence:
// one K tile and one V tile of those 160 rows feed both head tiles, and head tile t needs its
// rows 16 t .. 16 t + 143, so per head tile one S MMA of N = 144 covers the whole unit and each
// softmax thread exponentiates 144 columns of its row. (The general kernel tiles a window-128
// call as 128 queries x 2 key tiles of 128 for 2 heads: two masked steps per unit and 256
// exponentials per row.)
//
// Per CTA (384 threads, one CTA per SM, persistent over a static list of units; all units
// cost the same, so CTA c takes units c, c + grid, ...; consecutive CTAs take consecutive
// query blocks of one kv head at the same time, so their overlapping K/V spans come from L2):
//   warp 0      TMA producer of Q (both head tiles) and K
//   warp 2      TMA producer of V
//   warps 1, 3  MMA issuers of head tile 0 / 1: PV_t(u-1) then S_t(u), since P_t is written
//               over the first 72 columns of S_t (bf16 pairs)
//   warps 4-7   softmax of head tile 0, warps 8-11 of head tile 1; thread r owns row r
//               (TMEM lane r). Per unit: the exact row maximum of the visible columns, the
//               running maximum seeded with the head's sink (§Sink-Attention ¶3), P as bf16
//               into TMEM, the sum d including the sink's term. A unit is one step, so there
//               is no rescaling. The two warpgroups take turns (named barriers) from the TMEM
//               load of S to the P store; the epilogue (O / d as bf16, log-sum-exp) follows
//               PV_t(u) outside the turn.
// Output: each softmax warp stages its 32 rows (4 queries x 8 heads) in shared memory and
// writes them with one TMA store (box {64, 8, 4}), or with per-row stores past a sequence's end.
// TMEM (512 columns): head tile t has S_t (fp32, 144 columns) at 256 t, P_t (bf16 pairs, 72
// columns) over the first half of S_t, and O_t (fp32, 64 columns) at 256 t + 160.
// Every mbarrier wait is bounded; a timeout aborts the CTA cleanly through the same exits.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kQB = 32;      // queries per unit
constexpr int kQT = 16;      // queries per head tile (x 8 heads = 128 MMA rows)
constexpr int kSpan = 160;   // keys per unit: [q0 - 128, q0 + 32)
constexpr int kSN = 144;     // keys per head tile: span rows 16 t .. 16 t + 143
constexpr int kD = 64;       // head_dim
constexpr int kThreads = 384;
constexpr uint32_t kRegsLow = 72;    // producers and issuers
constexpr uint32_t kRegsHigh = 216;  // softmax warpgroups
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kNbTeardown = 1;
constexpr uint32_t kNbTurn = 2;  // + t: softmax warpgroup t may take its turn (256 threads)

// Turn hand-overs between the two softmax warpgroups carry no data (each touches only its own
// TMEM columns), so these forms do not clobber memory; being volatile they stay in order with
// the TMEM loads and stores around them.
__device__ __forceinline__ void turn_wait(uint32_t id) {
  asm volatile("bar.sync %0, 256;" ::"r"(id));
}
__device__ __forceinline__ void turn_pass(uint32_t id) {
  asm volatile("bar.arrive %0, 256;" ::"r"(id));
}

struct BandSmem {
  static constexpr int kQTile = 128 * 128;     // one head tile of Q (or O): 128 rows x 128 bytes
  static constexpr int kKVTile = kSpan * 128;  // one K or V span: 160 rows x 128 bytes
  static constexpr int kNQ = 2, kNK = 2, kNV = 2;
  static constexpr int kQ = 0;  // [kNQ][2 head tiles]
  static constexpr int kK = kQ + kNQ * 2 * kQTile;
  static constexpr int kV = kK + kNK * kKVTile;
  static constexpr int kO = kV + kNV * kKVTile;  // [2 head tiles]: output rows for the TMA store
  static constexpr int kBar = kO + 2 * kQTile;
  static constexpr int kBarQFull = 0, kBarQEmpty = kBarQFull + kNQ, kBarKFull = kBarQEmpty + kNQ,
                       kBarKEmpty = kBarKFull + kNK, kBarVFull = kBarKEmpty + kNK,
                       kBarVEmpty = kBarVFull + kNV, kBarSFull = kBarVEmpty + kNV,  // [2]
      kBarPFull = kBarSFull + 2,  // [2] P of keys 0..95 written, [2] P of keys 96..143 written
      kBarODone = kBarPFull + 4, kBarOFree = kBarODone + 2,
                       kBarDrain = kBarOFree + 2, kNumBars = kBarDrain + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base, [1] abort flag
  static constexpr int kPre = kMisc + 16;            // int [kBandMaxSeqs + 1]: query blocks
                                                     // of the sequences before s
  static constexpr int kList = (kPre + 4 * (kBandMaxSeqs + 1) + 15) / 16 * 16;  // int4 [units]
  static constexpr int kBytes = kList + kBandMaxUnits * 16 + 1024;  // + alignment slack
  static_assert(kQTile % 1024 == 0 && kKVTile % 1024 == 0, "1024-byte aligned stages");
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct BandParams {
  const int32_t* cu;  // [num_seqs + 1] query (and key) rows
  const float* sinks;
  __nv_bfloat16* out;
  float* lse;  // [T, Hq] natural log, or null
  unsigned* err;
  int num_seqs, T, max_seqlen, Hq, Hkv, G, window;
  int out32;  // `out` is 32-byte aligned: output rows are written with 32-byte stores
  float scale_log2;
  uint64_t timeout_ns;
};

// One unit of the CTA's list: row of the sequence's first query, its length, the unit's
// first query inside the sequence, and kv head | octet of query heads << 16. len == 0 marks
// an entry past the end of the work.
struct BandUnit {
  int start, len, q0, go;
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_band_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const BandParams p) {
  using S = BandSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t q_smem = sb + S::kQ, k_smem = sb + S::kK, v_smem = sb + S::kV;
  const uint32_t o_smem = sb + S::kO;
  auto bar = [&](int i) -> uint32_t { return sb + S::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);
  int* pre = reinterpret_cast<int*>(smem + S::kPre);
  int4* list = reinterpret_cast<int4*>(smem + S::kList);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kNumBars; ++i) {
      // Q, K and V stages are released by both issuers (one commit each); P written and O
      // read out are arrivals of the 128 softmax threads of a head tile.
      const bool by_threads = (i >= S::kBarPFull && i < S::kBarPFull + 4) ||
                              i == S::kBarOFree || i == S::kBarOFree + 1;
      const bool by_issuers = (i >= S::kBarQEmpty && i < S::kBarQEmpty + S::kNQ) ||
                              (i >= S::kBarKEmpty && i < S::kBarKEmpty + S::kNK) ||
                              (i >= S::kBarVEmpty && i < S::kBarVEmpty + S::kNV);
      mbar_init(bar(i), by_threads ? 128 : by_issuers ? 2 : 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (blockIdx.x == 0 && warp == 2) {
    for (int s = lane; s < p.num_seqs; s += 32) {
      const int a = p.cu[s], b = p.cu[s + 1];
      if (a < 0 || b < a || b > p.T || b - a > p.max_seqlen) atomicOr(p.err, kErrCuSeqlens);
    }
  }
  // ---- the CTA's unit list: query blocks of every sequence (malformed ones have none) ----
  if (warp == 0) {  // exclusive prefix of the sequences' block counts, 32 contiguous runs
    const int per_lane = (p.num_seqs + 31) / 32;
    const int s_lo = lane * per_lane, s_hi = min(s_lo + per_lane, p.num_seqs);
    int sum = 0;
    for (int s = s_lo; s < s_hi; ++s) {
      const int a = p.cu[s], b = p.cu[s + 1];
      sum += (a < 0 || b < a || b > p.T) ? 0 : (b - a + kQB - 1) / kQB;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += x;
    }
    int run = incl - sum;
    for (int s = s_lo; s < s_hi; ++s) {
      pre[s] = run;
      const int a = p.cu[s], b = p.cu[s + 1];
      run += (a < 0 || b < a || b > p.T) ? 0 : (b - a + kQB - 1) / kQB;
    }
    if (lane == 31) pre[p.num_seqs] = incl;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const int n_blocks = pre[p.num_seqs];
  const int n_oct = p.G / 8;
  const int n_units = n_blocks * p.Hkv * n_oct;
  const int n_list = min((n_units + (int)gridDim.x - 1) / (int)gridDim.x, kBandMaxUnits);
  for (int i = threadIdx.x; i < n_list; i += kThreads) {
    // kv head and octet slowest, query blocks fastest: CTAs working at the same time take
    // neighbouring blocks, whose key spans overlap.
    const int k = i * (int)gridDim.x + (int)blockIdx.x;
    int4 e = make_int4(0, 0, 0, 0);
    if (k < n_units) {
      const int og = k / n_blocks, blk = k - og * n_blocks;
      int lo = 0, hi = p.num_seqs;  // last sequence with pre[s] <= blk
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= blk) lo = mid; else hi = mid;
      }
      const int a = p.cu[lo], b = p.cu[lo + 1];
      e = make_int4(a, b - a, (blk - pre[lo]) * kQB, (og / n_oct) | ((og % n_oct) << 16));
    }
    list[i] = e;
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  auto unit_at = [&](int i) -> BandUnit {
    const int4 e = list[i];
    return BandUnit{e.x, e.y, e.z, e.w};
  };
  static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * 168, "register split");

  if (warp < 4) {
    regs_dealloc<kRegsLow>();
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
    };
    if (warp == 0 || warp == 2) {
      // ============ TMA producers: warp 0 loads Q and K, warp 2 loads V ============
      // Per unit: Q of both head tiles (heads h .. h+7 of queries q0 .. q0+15 and of q0+16 ..
      // q0+31) and the 160-row K span, or the V span. Rows before the first row or past the last
      // one are filled with zeros by the copy; rows of a neighbouring sequence are masked.
      const bool qk = warp == 0;
      if (elect_one()) {
        if (qk) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
        } else {
          tma_prefetch_desc(&tm_v);
        }
      }
      int qc = 0, kc = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_list; ++i) {
        const BandUnit u = unit_at(i);
        if (u.len == 0) continue;
        const int g = u.go & 0xffff, h0 = g * p.G + 8 * (u.go >> 16);
        const int krow = u.start + u.q0 - 128;
        if (qk) {
          const int qs = qc % S::kNQ;
          if (!(ok = wait(bar(S::kBarQEmpty + qs), ((qc / S::kNQ) & 1) ^ 1))) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(S::kBarQFull + qs), 2 * S::kQTile);
            for (int t = 0; t < 2; ++t)
              tma_load_3d(q_smem + (2 * qs + t) * S::kQTile, &tm_q, bar(S::kBarQFull + qs), 0,
                          h0, u.start + u.q0 + kQT * t);
          }
          __syncwarp();
          ++qc;
        }
        const int ks = kc % S::kNK;  // (the V ring has the same depth)
        const uint32_t empty = qk ? bar(S::kBarKEmpty + ks) : bar(S::kBarVEmpty + ks);
        const uint32_t full = qk ? bar(S::kBarKFull + ks) : bar(S::kBarVFull + ks);
        if (!(ok = wait(empty, ((kc / S::kNK) & 1) ^ 1))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(full, S::kKVTile);
          tma_load_3d((qk ? k_smem : v_smem) + ks * S::kKVTile, qk ? &tm_k : &tm_v, full, 0, g,
                      krow);
        }
        __syncwarp();
        ++kc;
      }
      static_assert(S::kNK == S::kNV, "K and V rings are walked by one counter each");
      // Let every copy still in flight land before the CTA may exit.
      if (lane == 0) {
        for (int i = max(0, kc - S::kNK); i < kc; ++i)
          mbar_drain(qk ? bar(S::kBarKFull + i % S::kNK) : bar(S::kBarVFull + i % S::kNK),
                     (i / S::kNK) & 1, p.timeout_ns);
        for (int i = max(0, qc - S::kNQ); i < qc; ++i)
          mbar_drain(bar(S::kBarQFull + i % S::kNQ), (i / S::kNQ) & 1, p.timeout_ns);
      }
    } else {
      // ============ MMA issuers: warp 1 for head tile 0, warp 3 for head tile 1 ============
      // Per unit u: PV_t(u-1) (P_t(u-1) written, V resident, O_t read out by the epilogue of
      // u-2), then S_t(u) = Q_t K^T (M = 128, N = 144, K = 64) into S_t, with K rows 16 t ..
      // 16 t + 143 of the span (whole 1024-byte swizzle atoms from the tile's start).
      const int t = warp == 1 ? 0 : 1;
      constexpr uint32_t idS = idesc_bf16_f32(128, kSN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, kD, false, true);
      constexpr uint32_t hi = sdesc_sw128_hi(1024);
      const uint32_t lo_q0 = sdesc_sw128_lo(q_smem, 16);
      const uint32_t lo_k0 = sdesc_sw128_lo(k_smem, 16);
      const uint32_t lo_v0 = sdesc_sw128_lo(v_smem, 16384);
      const uint32_t dS = tmem + 256u * t, dO = dS + 160, aP = dS;
      const uint32_t span_off = (uint32_t)(kQT * 128 * t) >> 4;  // rows 16 t.. of K and V
      int qc = 0, kc = 0, vc = 0, n = 0;
      bool ok = true;
      auto do_pv = [&](int j) -> bool {  // PV_t of this tile's unit number j
        const int vs = vc % S::kNV;
        if (!wait(bar(S::kBarVFull + vs), (vc / S::kNV) & 1)) return false;
        if (j > 0 && !wait(bar(S::kBarOFree + t), (j - 1) & 1)) return false;
        // P arrives in two parts (keys 0..95, then 96..143), so the first six MMAs run while
        // the softmax still computes the last 48 columns.
        if (!wait(bar(S::kBarPFull + t), j & 1)) return false;
        tc_fence_after_sync();
        const uint32_t bv = lo_v0 + vs * (S::kKVTile >> 4) + span_off;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 6; ++kk)  // 16 keys (2048 bytes of V) per MMA
            umma_ts(dO, aP + kk * 8, sdesc_join(bv + kk * (2048 >> 4), hi), idPV, kk > 0 ? 1u : 0u);
        }
        __syncwarp();
        if (!wait(bar(S::kBarPFull + 2 + t), j & 1)) return false;
        tc_fence_after_sync();
        if (elect_one()) {
#pragma unroll
          for (int kk = 6; kk < kSN / 16; ++kk)
            umma_ts(dO, aP + kk * 8, sdesc_join(bv + kk * (2048 >> 4), hi), idPV, 1u);
          umma_commit(bar(S::kBarODone + t));
          umma_commit(bar(S::kBarVEmpty + vs));
        }
        __syncwarp();
        ++vc;
        return true;
      };
      for (int i = 0; ok && i < n_list; ++i) {
        if (list[i].y == 0) continue;
        if (n > 0 && !(ok = do_pv(n - 1))) break;
        const int qs = qc % S::kNQ, ks = kc % S::kNK;
        if (!(ok = wait(bar(S::kBarQFull + qs), (qc / S::kNQ) & 1))) break;
        if (!(ok = wait(bar(S::kBarKFull + ks), (kc / S::kNK) & 1))) break;
        tc_fence_after_sync();
        const uint32_t aq = lo_q0 + (2 * qs + t) * (S::kQTile >> 4);
        const uint32_t bk = lo_k0 + ks * (S::kKVTile >> 4) + span_off;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)  // 32 bytes of each row per K = 16 step
            umma_ss(dS, sdesc_join(aq + kk * 2, hi), sdesc_join(bk + kk * 2, hi), idS,
                    kk > 0 ? 1u : 0u);
          umma_commit(bar(S::kBarSFull + t));
          umma_commit(bar(S::kBarKEmpty + ks));
          umma_commit(bar(S::kBarQEmpty + qs));
        }
        __syncwarp();
        ++qc;
        ++kc;
        ++n;
      }
      if (ok && n > 0) ok = do_pv(n - 1);
      // Wait for every MMA this warp issued before TMEM can be released.
      if (elect_one()) {
        umma_commit(bar(S::kBarDrain + t));
        mbar_drain(bar(S::kBarDrain + t), 0, p.timeout_ns);
      }
      __syncwarp();
    }
    __syncwarp();
    tc_fence_before_sync();
    named_barrier_sync(kNbTeardown, kThreads);  // every warp of the CTA is done with TMEM
    if (warp == 1) {
      tc_fence_after_sync();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    // ============================ softmax warpgroups ============================
    regs_alloc<kRegsHigh>();
    const int t = (warp - 4) >> 2;  // head tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row = quarter * 32 + lane;
    const int tok = row >> 3, hs = row & 7;  // row = 8 * query + head
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + 256u * t;
    const uint32_t ts = tl, tp = tl, to = tl + 160;
    const float sl = p.scale_log2;
    const float2 sl2 = make_float2(sl, sl);
    // The two warpgroups take turns through named barriers: a turn runs from the TMEM load of
    // S to the P store, so one warpgroup's exponentials overlap the other's PV and epilogue
    // instead of both contending for the same units at the same time.
    if (t == 1) turn_pass(kNbTurn + 0);  // warpgroup 0 goes first
    int n = 0;
    int i = 0, stage = 2;  // position for the dry tail: 0 turn not taken, 1 taken, 2 handed over
    bool ok = true;
    for (; ok && i < n_list; ++i) {
      const BandUnit u = unit_at(i);
      if (u.len == 0) continue;
      stage = 0;
      const int h = (u.go & 0xffff) * p.G + 8 * (u.go >> 16) + hs;
      const int qt = u.q0 + kQT * t;  // the head tile's first query inside its sequence
      const int qi = qt + tok;        // this row's query
      const float m0 = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarSFull + t), n & 1, wc)))) break;
      turn_wait(kNbTurn + t);  // the other warpgroup's turn is over
      stage = 1;
      tc_fence_after_sync();
      uint32_t r[kSN];
      tmem_ld144(ts, r);
      float s[kSN];
#pragma unroll
      for (int c = 0; c < kSN; ++c) s[c] = __uint_as_float(r[c]);
      // Column c holds key position qt - 128 + c; visible: lo <= c <= hi (the key at or before
      // the query, inside the window, and not before the sequence's first row).
      const int hi = tok + 128;
      const int lo = max(128 - qt, tok + 129 - p.window);
      // Columns 16..127 are visible to every row of the tile when the window is 128 keys and
      // its keys start at or after the sequence's first row plus 16 (qt >= 112): then only the
      // first and the last 16 columns are masked.
      const bool mid_visible = qt >= 112 && p.window >= 128;
      // One visibility word per 16 columns, then one bit test per column.
#pragma unroll
      for (int b = 0; b < kSN / 16; ++b) {
        if (b != 0 && b != kSN / 16 - 1 && mid_visible) continue;
        const int hc = min(max(hi, 16 * b - 1), 16 * b + 15) - 16 * b;  // -1 .. 15
        const int lc = min(max(lo, 16 * b), 16 * b + 16) - 16 * b;      // 0 .. 16
        const uint32_t vis =
            hc >= lc ? (0xffffu >> (15 - hc)) & (0xffffu << lc) : 0u;  // bits lc..hc
#pragma unroll
        for (int c = 0; c < 16; ++c) s[16 * b + c] = (vis & (1u << c)) ? s[16 * b + c] : -INFINITY;
      }
      // Row maximum of the visible columns: 8 independent three-input chains, then 8 -> 1.
      float mp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mp[a] = fmaxf(s[a], s[8 + a]);
#pragma unroll
      for (int c = 16; c < kSN; c += 16) {
#pragma unroll
        for (int a = 0; a < 8; ++a) mp[a] = fmax3(mp[a], s[c + a], s[c + 8 + a]);
      }
      const float mx =
          fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      const float m = fmaxf(m0, mx * sl);
      const float mu = (m == -INFINITY) ? 0.f : m;
      const float2 nmu = make_float2(-mu, -mu);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};  // independent partial row sums
      // P over S_t's columns, all of which are already in registers: four blocks of 32
      // columns (16 packed words) and one of 16.
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = 32 * c4 + 2 * e;
          const float2 x = ffma2(make_float2(s[c], s[c + 1]), sl2, nmu);
          const float2 pe = make_float2(ex2(x.x), ex2(x.y));
          acc[e & 3] = fadd2(acc[e & 3], pe);
          pk[e] = pack_bf16x2(pe.x, pe.y);
        }
        tmem_st16(tp + 16 * c4, pk);
        if (c4 == 2) {  // keys 0..95 written: the first six PV MMAs may start
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(bar(S::kBarPFull + t));
        }
      }
      {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 128 + 2 * e;
          const float2 x = ffma2(make_float2(s[c], s[c + 1]), sl2, nmu);
          const float2 pe = make_float2(ex2(x.x), ex2(x.y));
          acc[e & 3] = fadd2(acc[e & 3], pe);
          pk[e] = pack_bf16x2(pe.x, pe.y);
        }
        tmem_st8(tp + 64, pk);
      }
      turn_pass(kNbTurn + (t ^ 1));
      stage = 2;
      const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
      const float d = ex2(m0 - mu) + ((a01.x + a23.x) + (a01.y + a23.y));  // the sink's term
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(S::kBarPFull + 2 + t));
      // ---- epilogue: O / d -> bf16 once PV_t(u) is done, rows of this sequence only ----
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarODone + t), n & 1, wc)))) break;
      tc_fence_after_sync();
      const float inv = d > 0.f ? 1.f / d : 0.f;
      const bool row_ok = qi < u.len;
      const size_t orow = (size_t)(u.start + qi) * p.Hq + h;
      if (u.len - (qt + 4 * quarter) >= 4) {
        // The warp's 4 queries (x 8 heads) all in the sequence: its 32 rows go to its 4 KB of
        // shared memory in the layout of the output box (row = 8 * query + head, 128-byte
        // swizzle) and leave in one TMA store of the warp, instead of 32 stores of 128 bytes.
        const uint32_t wbuf = o_smem + t * S::kQTile + quarter * 4096;
        if (lane == 0) bulk_wait_group_read0();  // the warp's previous store has read wbuf
        __syncwarp();
        uint32_t o[kD];
        tmem_ld64(to, o);
#pragma unroll
        for (int c4 = 0; c4 < kD / 32; ++c4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t w4[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2)
              w4[k2] = pack_bf16x2(__uint_as_float(o[32 * c4 + 8 * e + 2 * k2]) * inv,
                                   __uint_as_float(o[32 * c4 + 8 * e + 2 * k2 + 1]) * inv);
            const int chunk = 4 * c4 + e;  // 16-byte chunk of the 128-byte row
            const uint32_t a = wbuf + lane * 128 + ((chunk ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w4[0]),
                         "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                         : "memory");
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, wbuf, 0, (u.go & 0xffff) * p.G + 8 * (u.go >> 16),
                       u.start + qt + 4 * quarter);
          bulk_commit_group();
        }
      } else {
        // Queries past the sequence's last row: per-row stores, rows of this sequence only.
        uint4* dst = reinterpret_cast<uint4*>(p.out + (row_ok ? orow : 0) * kD);
#pragma unroll
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(to + 32 * c4, o);
          uint32_t q16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            q16[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          if (row_ok) {
            if (p.out32) {
#pragma unroll
              for (int e = 0; e < 2; ++e) st_global_v8(dst + c4 * 4 + 2 * e, &q16[8 * e]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[c4 * 4 + e] = make_uint4(q16[4 * e], q16[4 * e + 1], q16[4 * e + 2], q16[4 * e + 3]);
            }
          }
        }
      }
      // log-sum-exp of the row: m and d are in the scaled exp2 domain (d relative to m)
      if (p.lse && row_ok)
        p.lse[orow] = (d > 0.f && m != -INFINITY) ? (m + log2f(d)) * kLn2 : -INFINITY;
      tc_fence_before_sync();
      mbar_arrive(bar(S::kBarOFree + t));
      ++n;
    }
    if (!ok) {
      // Dry tail: the remaining turn hand-overs of this warpgroup's list, all blocking, so
      // that the partner warpgroup (which aborts as well, its waits seeing the abort flag)
      // never waits on a turn that does not come.
      for (; i < n_list; ++i, stage = 0) {
        if (list[i].y == 0) continue;
        if (stage < 1) turn_wait(kNbTurn + t);
        if (stage < 2) turn_pass(kNbTurn + (t ^ 1));
      }
    }
    // Warpgroup 1's hand-overs lead warpgroup 0's turns by one: take the last.
    if (t == 0) turn_wait(kNbTurn + 0);
    if (lane == 0) bulk_wait_group0();  // the warp's output stores are complete
    __syncwarp();
    tc_fence_before_sync();
    named_barrier_sync(kNbTeardown, kThreads);
  }
}

}  // namespace

cudaError_t launch_prefill_band(const PrefillLaunch& a, cudaStream_t stream) {
  using S = BandSmem;
  BandParams p{};
  p.cu = a.cu_seqlens;
  p.sinks = a.sinks;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.out32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
  p.lse = a.lse;
  p.err = a.err;
  p.num_seqs = a.num_seqs;
  p.T = a.total_tokens;
  p.max_seqlen = a.max_seqlen;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.G = a.num_q_heads / a.num_kv_heads;
  p.window = a.window;
  p.scale_log2 = a.scale * kLog2e;
  p.timeout_ns = a.timeout_ns;
  cudaError_t e =
      cudaFuncSetAttribute(prefill_band_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (e != cudaSuccess) return e;
  prefill_band_kernel<<<a.num_sms, kThreads, S::kBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o,
                                                                  p);
  return cudaGetLastError();
}

}  // namespace sa
