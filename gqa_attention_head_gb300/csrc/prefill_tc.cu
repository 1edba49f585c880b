// prefill_tc.cu — ragged causal (optionally sliding-window) prefill with a per-head
// sink logit on sm_103a tensor cores.
//
// Work decomposition: a persistent grid walks work units (q tile of 128 rows,
// sequence, kv head, pair of query heads of that kv head's group), the last q tiles
// of the longest sequences first (they see the most keys); units of one kv head are
// adjacent so their K/V tiles are shared through L2. The two query heads of a unit
// read the same K/V tiles under the same mask, so every K/V tile staged in shared
// memory feeds two S MMAs and two PV MMAs. Attention is parallel over heads and over
// the key sequence ("GPT-OSS am Day 0", §Sink-Attention ¶2); prefill is compute-bound
// ("Qwen hosten op Blackwell", §Prefillers).
//
// Per CTA (384 threads = 3 warpgroups, one CTA per SM). The kernel is launched with
// 168 registers per thread; warpgroup 0 keeps 96 each and the two softmax warpgroups
// take 192 each: 128*96 + 256*192 <= 384*168. No function
// called from the split regions may be out of line (one body cannot serve both
// register limits), so every helper is inlined.
// Warpgroup 0 (producers and MMA issuers; every role walks the schedule with the whole
// warp and issues from one elected lane):
//   head_dim 64  warp 0 loads Q (a ring of Q stages, each holding the unit's two head
//                tiles), K and V; warp 1 issues S_t = Q_t K^T (M=128, N=128, K=64) for both
//                head tiles into TMEM S_t; warps 2 and 3 issue O_t += P_t V (M=128, N=64,
//                K=128) for head tile 0 and 1, with P_t read from TMEM. A PV issuer waits for
//                nothing but V and the softmax's "P written", so the PV follows it directly.
//   head_dim 128 warp 0 loads Q and K, warp 2 loads V (its own ring, so K never waits
//                behind V); warps 1 and 3 each issue both MMAs of one head tile, in the order
//                PV_t(j-1) then S_t(j), because P_t overwrites S_t's columns.
//   paged K/V at head_dim 64 takes the head_dim-128 roles, with S_t(j+1) issued before
//                PV_t(j) (P_t has its own columns there).
// All stages are 128-byte swizzled; warp 1 allocates the 512 TMEM columns.
// Warps 4-7 are the softmax warpgroup of head tile 0, warps 8-11 that of head tile 1;
// thread r owns row r (TMEM lane r): masks, runs the online softmax in the exp2 domain
// with the running maximum seeded by the head's sink ("GPT-OSS am Day 0",
// §Sink-Attention ¶3), writes P as bf16 to TMEM, rescales O only when some row's maximum
// grew by more than 2^8, and stores O / d as bf16.
//
// When every unit has both head tiles (an even group size), the two softmax warpgroups
// take turns: a warpgroup's turn starts before its TMEM load of S and, at head_dim 128,
// ends after its exponentials (each warpgroup then has the MUFU unit to itself); at
// head_dim 64 the hand-over is left unordered against the exponentials, which measured
// faster there. The hand-over is a named barrier (a few tens of cycles, against about
// 150 for an mbarrier arrive/wait pair on this part).
//
// Every mbarrier wait is bounded (see sm103_ptx.cuh); a timeout aborts the CTA cleanly.
// A softmax warp that aborts does not leave while its partner warpgroup could still
// wait for a turn: it finishes its schedule "dry", performing only the remaining turn
// hand-overs, all as blocking bar.sync, so every bar.sync meets its partner and no
// barrier ever receives arrivals for two phases at once.
#include <limits.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr int kPageRows = 16;  // tokens per page of the paged cache (8 pages per key tile)
constexpr int kThreads = 384;
constexpr uint32_t kRegsLow = 96;    // warpgroup 0 (producers, MMA issuers)
constexpr uint32_t kRegsHigh = 192;  // softmax warpgroups
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Named barriers (0 is __syncthreads).
constexpr uint32_t kNbTeardown = 1;  // all threads
constexpr uint32_t kNbTurn = 2;      // + t: softmax warpgroup t may take its turn (256 threads)
// Work schedule: the valid units, longest first, dealt to the CTAs in a snake order
// (round r goes left to right when r is even, right to left when odd), which balances
// the causal cost much better than plain round-robin. Its shared-memory tables cap the
// sizes it handles; beyond them every CTA falls back to round-robin over all unit ids.
constexpr int kMaxSchedSeqs = 128;
constexpr int kMaxSchedQTiles = 512;
constexpr int kMaxSortPairs = 4096;  // (q tile, sequence) pairs the unit list sorts at most

// TMEM columns (512 allocated). S_t (fp32, 128 columns) at [128 t, 128 t + 128).
// head_dim 64: P_t (bf16 pairs, 64 columns) has its own columns at 256 + 64 t and O_t
// is at 384 + 64 t, so S_t(j+1) can be computed while the softmax still works on
// P_t(j). head_dim 128: 2 S + 2 O use all 512 columns, P_t overwrites the first 64
// columns of S_t, and S_t(j+1) has to wait until PV_t(j) has been issued.
template <int D>
struct TmemCols {
  static constexpr bool kSepP = (D == 64);
  static constexpr uint32_t s(int t) { return 128u * t; }
  static constexpr uint32_t p(int t) { return kSepP ? 256u + 64u * t : 128u * t; }
  static constexpr uint32_t o(int t) { return kSepP ? 384u + 64u * t : 256u + (uint32_t)D * t; }
};

template <int D>
struct PrefillSmem {
  static constexpr int kBoxes = D / 64;            // 64-element (128-byte) column blocks
  static constexpr int kBoxBytes = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;   // one Q, K or V tile
  static constexpr int kNQ = (D == 64) ? 2 : 1;    // Q ring depth (a stage holds both head tiles)
  static constexpr int kNK = (D == 64) ? 4 : 2;    // K ring depth (head_dim 128: 3 -> 2 measured
                                                   // 0.5% faster and frees room for the unit list)
  static constexpr int kNV = (D == 64) ? 4 : 2;    // V ring depth
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kNQ * 2 * kTileBytes;
  static constexpr int kV = kK + kNK * kTileBytes;
  static constexpr int kBar = kV + kNV * kTileBytes;
  static constexpr int kBarQFull = 0, kBarQEmpty = kBarQFull + kNQ, kBarKFull = kBarQEmpty + kNQ,
                       kBarKEmpty = kBarKFull + kNK, kBarVFull = kBarKEmpty + kNK,
                       kBarVEmpty = kBarVFull + kNV,
                       kBarSFull = kBarVEmpty + kNV,  // [2] per head tile
      kBarSFree = kBarSFull + 2, kBarPFull = kBarSFree + 2, kBarODone = kBarPFull + 2,
                       kBarOFree = kBarODone + 2, kBarDrain = kBarOFree + 2,  // [3]
                       kNumBars = kBarDrain + 3;
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base, [1] abort flag
  static constexpr int kOrd = kMisc + 16;              // uint8 [kMaxSchedSeqs]
  static constexpr int kPre = kOrd + kMaxSchedSeqs;    // uint16 [kMaxSchedQTiles + 1]
  // Windowed head_dim 64: each softmax thread's pending epilogue (row, 1/d, log-sum-exp).
  static constexpr int kPend = (kPre + 2 * (kMaxSchedQTiles + 1) + 15) / 16 * 16;
  static constexpr int kPendBytes = (D == 64) ? 2 * 128 * 16 : 0;
  // The CTA's units, decoded once at the start (48 bytes each). Window 128: 152 -> 129 us,
  // causal 0.765 -> 0.743 ms, Qwen3-235B-style head_dim 128 0.741 -> 0.735 ms: the lookup and
  // the row-offset loads sat in every unit start.
  // (Addressing the list through a 32-bit shared address moved the kernel's few spilled
  // registers into the step loop and lost the gain: 0.764 ms.)
  static constexpr int kMaxListUnits = 512;
  static constexpr int kList = (kPend + kPendBytes + 15) / 16 * 16;
  static constexpr int kBytes = kList + kMaxListUnits * 48 + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct PrefillParams {
  const int32_t* cu;       // [num_seqs + 1] query rows (and, contiguous, key rows)
  const int32_t* cu_k;     // contiguous, keys apart from queries: [num_seqs + 1] key rows;
                           // the queries are the last rows of their key range; else null
  int Tk;                  // with cu_k: rows of K and V
  const int32_t* kv_lens;  // paged: [num_seqs] keys per sequence after the append; else null
  const int32_t* page_table;  // paged: [num_seqs][max_pages]
  int max_pages, num_pages, max_kv;
  const float* sinks;
  __nv_bfloat16* out;
  float* lse;  // [T, Hq] natural log, or null
  unsigned* err;
  int num_seqs, T, max_seqlen, Hq, Hkv, G, npairs, window, n_qt, total_units;
  int snake;     // use the snake schedule (sizes within its table caps)
  int pingpong;  // every unit has both head tiles: the softmax warpgroups take turns
  int out32;     // `out` is 32-byte aligned: output rows are written with 32-byte stores
  float scale_log2;
  uint64_t timeout_ns;
};

struct Unit {
  int start, L, q0, g, h0, has1, kv_lo, n_kv;
  int s;       // sequence index
  int Lk;      // keys of the sequence (paged: cache length after the append; with cu_k its
               // key rows; else L)
  int off;     // key position of query row 0: Lk - L (0 when queries and keys coincide)
};

// Fill unit (q tile index qi from the end, sequence s, kv head g, head pair pr).
// Returns false for units with no rows (or a malformed sequence).
template <bool KVOWN>
__device__ __forceinline__ bool decode_unit(const PrefillParams& p, int qi, int s, int g, int pr,
                                            Unit& w) {
  w.g = g;
  w.h0 = w.g * p.G + 2 * pr;
  w.has1 = (2 * pr + 1 < p.G) ? 1 : 0;
  const int start = p.cu[s], end = p.cu[s + 1];
  if (start < 0 || end < start || end > p.T) return false;
  w.start = start;
  w.L = end - start;
  w.s = s;
  w.Lk = w.L;
  if (p.kv_lens) {  // chunked prefill over the paged cache: the new rows are the last ones
    w.Lk = p.kv_lens[s];
    if (w.Lk < w.L || w.Lk > p.max_kv || (w.Lk + kPageRows - 1) / kPageRows > p.max_pages)
      return false;
  } else if constexpr (KVOWN) {  // contiguous keys of their own: queries are the last rows
    const int ka = p.cu_k[s], kb = p.cu_k[s + 1];
    if (ka < 0 || kb < ka || kb > p.Tk || kb - ka < w.L || kb - ka > p.max_kv) return false;
    w.Lk = kb - ka;
  }
  w.off = w.Lk - w.L;
  w.q0 = (p.n_qt - 1 - qi) * kBM;
  if (w.q0 >= w.L) return false;
  const int q1 = min(w.q0 + kBM, w.L);
  const int kv_hi = (w.off + q1 + kBN - 1) / kBN;
  w.kv_lo = (p.window > 0) ? max(0, w.off + w.q0 - p.window + 1) / kBN : 0;
  w.n_kv = kv_hi - w.kv_lo;
  return true;
}

// Unit id u of the full (qi, s, g, pr) enumeration.
template <bool KVOWN>
__device__ __forceinline__ bool unit_info(const PrefillParams& p, int u, Unit& w) {
  const int per_s = p.Hkv * p.npairs;
  const int per = p.num_seqs * per_s;
  const int qi = u / per;
  int rem = u - qi * per;
  const int s = rem / per_s;
  rem -= s * per_s;
  const int g = rem / p.npairs;
  return decode_unit<KVOWN>(p, qi, s, g, rem - g * p.npairs, w);
}

// The CTA's sequence of units (identical for every role of the CTA).
struct UnitSched {
  const uint8_t* ord;    // sequences by decreasing length
  const uint16_t* pre;   // pre[qi] = sequence-units of q-tile indices < qi
  int total;             // valid units (snake) or all unit ids (round-robin)
  int snake;
  const int4* list;      // LIST: the CTA's units decoded in shared memory (3 int4 each)
  int n_list;
};

// Unit (kv head, head pair) number rem of (q tile, sequence) pair ks of the snake order.
template <bool KVOWN>
__device__ __forceinline__ bool pair_unit(const PrefillParams& p, const UnitSched& sc, int ks,
                                          int rem, Unit& w) {
  int lo = 0, hi = p.n_qt;  // largest qi with pre[qi] <= ks
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sc.pre[mid] <= ks) lo = mid; else hi = mid;
  }
  const int g = rem / p.npairs;
  return decode_unit<KVOWN>(p, lo, sc.ord[ks - sc.pre[lo]], g, rem - g * p.npairs, w);
}

// Unit k of the snake list (k < total).
template <bool KVOWN>
__device__ __forceinline__ bool snake_unit(const PrefillParams& p, const UnitSched& sc, int k,
                                           Unit& w) {
  const int per_s = p.Hkv * p.npairs;
  const int ks = k / per_s;
  return pair_unit<KVOWN>(p, sc, ks, k - ks * per_s, w);
}

// The CTA's next unit after round r (advances r). LIST: read from the list decoded in
// shared memory at the start (units without rows are stored invalid and skipped); else
// decoded here, which costs a lookup and dependent loads of row offsets at every unit.
template <bool KVOWN, bool LIST>
__device__ __forceinline__ bool next_unit(const PrefillParams& p, const UnitSched& sc, int& r,
                                          Unit& w) {
  if constexpr (LIST) {
    while (r < sc.n_list) {
      const int4* u = sc.list + 3 * r++;
      const int4 a = u[0], b = u[1], e = u[2];
      if (e.w) {
        w.start = a.x; w.L = a.y; w.q0 = a.z; w.g = a.w;
        w.h0 = b.x; w.has1 = b.y; w.kv_lo = b.z; w.n_kv = b.w;
        w.s = e.x; w.Lk = e.y; w.off = e.z;
        return true;
      }
    }
    return false;
  }
  const int G = gridDim.x, c = blockIdx.x;
  while (true) {
    const int base = r * G;
    if (base >= sc.total) return false;
    const int k = base + (sc.snake && (r & 1) ? G - 1 - c : c);
    ++r;
    if (k >= sc.total) continue;
    if (sc.snake ? snake_unit<KVOWN>(p, sc, k, w) : unit_info<KVOWN>(p, k, w)) return true;
  }
}

template <int D, bool PAGED, bool KVOWN, bool DEFER, bool LIST>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using S = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t q_smem = sb + S::kQ, k_smem = sb + S::kK, v_smem = sb + S::kV;
  auto bar = [&](int i) -> uint32_t { return sb + S::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kNumBars; ++i) {
      const bool by_threads = (i == S::kBarPFull || i == S::kBarPFull + 1 ||
                               i == S::kBarOFree || i == S::kBarOFree + 1 ||
                               i == S::kBarSFree || i == S::kBarSFree + 1);
      // Stages released by two issuing warps (barrier count 2): head_dim 64 has one S
      // issuer (Q and K stages, count 1) and one PV issuer per head tile (V stages);
      // head_dim 128 has one issuer per head tile for everything.
      const bool q_or_k = (i >= S::kBarQEmpty && i < S::kBarQEmpty + S::kNQ) ||
                          (i >= S::kBarKEmpty && i < S::kBarKEmpty + S::kNK);
      const bool by_issuers = ((!TmemCols<D>::kSepP || PAGED) && q_or_k) ||
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
      if (PAGED) {
        const int lk = p.kv_lens[s];
        if (lk < b - a || lk > p.max_kv || (lk + kPageRows - 1) / kPageRows > p.max_pages)
          atomicOr(p.err, kErrSeqLen);
      } else if (KVOWN) {
        const int ka = p.cu_k[s], kb = p.cu_k[s + 1];
        if (ka < 0 || kb < ka || kb > p.Tk) atomicOr(p.err, kErrCuSeqlens);
        else if (kb - ka < b - a || kb - ka > p.max_kv) atomicOr(p.err, kErrSeqLen);
      }
    }
  }
  // ---- schedule tables (built by every CTA; the K ring is free scratch until then) ----
  uint8_t* ord = smem + S::kOrd;
  uint16_t* pre = reinterpret_cast<uint16_t*>(smem + S::kPre);
  int* lens = reinterpret_cast<int*>(smem + S::kK);
  int* nval = lens + kMaxSchedSeqs;
  if (p.snake) {
    for (int s = threadIdx.x; s < p.num_seqs; s += kThreads) {
      const int a = p.cu[s], b = p.cu[s + 1];
      lens[s] = (a < 0 || b < a || b > p.T) ? 0 : b - a;
    }
    __syncthreads();
    for (int s = threadIdx.x; s < p.num_seqs; s += kThreads) {
      int rank = 0;
      for (int s2 = 0; s2 < p.num_seqs; ++s2)
        rank += (lens[s2] > lens[s]) || (lens[s2] == lens[s] && s2 < s);
      ord[rank] = (uint8_t)s;
    }
    for (int qi = threadIdx.x; qi < p.n_qt; qi += kThreads) {
      const int q0 = (p.n_qt - 1 - qi) * kBM;
      int n = 0;
      for (int s2 = 0; s2 < p.num_seqs; ++s2) n += lens[s2] > q0;
      nval[qi] = n;
    }
    __syncthreads();
    if (warp == 0) {  // prefix sums over q-tile indices, 32 contiguous blocks
      const int per_lane = (p.n_qt + 31) / 32;
      const int q_lo = lane * per_lane, q_hi = min(q_lo + per_lane, p.n_qt);
      int sum = 0;
      for (int qi = q_lo; qi < q_hi; ++qi) sum += nval[qi];
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += x;
      }
      int run = incl - sum;
      for (int qi = q_lo; qi < q_hi; ++qi) {
        pre[qi] = (uint16_t)run;
        run += nval[qi];
      }
      if (lane == 31) pre[p.n_qt] = (uint16_t)incl;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const int total_units = p.snake ? (int)pre[p.n_qt] * p.Hkv * p.npairs : p.total_units;
  UnitSched sched{ord, pre, total_units, p.snake, nullptr, 0};
  {
    // Decode the CTA's whole unit list at once (one unit per thread), so that no role pays
    // the schedule lookup and the dependent row-offset loads at each unit start.
    const int n_list = (total_units + (int)gridDim.x - 1) / (int)gridDim.x;
    if constexpr (LIST) {  // the host checked that the snake list fits
      // Paged and separate-key launches: the sequences' cached prefixes differ, so the
      // units' key-tile counts do not follow the snake order (q tiles from the end,
      // sequences by length). The (q tile, sequence) pairs are then sorted by their key-tile
      // count, longest first, with a bitonic sort in the K ring (unused until the producers
      // start), so that the snake deal can balance them: chunked gpt-oss prefill 0.942 ->
      // 0.978 of a perfect balance, simulated. Causal contiguous launches are in that order
      // already.
      const int per_s = p.Hkv * p.npairs;
      const int n_pairs = total_units / per_s;
      int npad = 1;
      while (npad < n_pairs) npad <<= 1;
      unsigned long long* key = reinterpret_cast<unsigned long long*>(smem + S::kK + 4096);
      static_assert(4096 + 8 * kMaxSortPairs <= S::kNK * S::kTileBytes,
                    "the pair keys must fit in the K ring");
      const bool sorted = (PAGED || KVOWN) && npad <= kMaxSortPairs;
      if (sorted) {
        for (int j = threadIdx.x; j < npad; j += kThreads) {
          unsigned long long kk = ~0ull;
          if (j < n_pairs) {
            Unit w{};
            const unsigned n = pair_unit<KVOWN>(p, sched, j, 0, w) ? (unsigned)w.n_kv : 0u;
            kk = ((unsigned long long)(0xffffffffu - n) << 32) | (unsigned)j;
          }
          key[j] = kk;
        }
        for (int size = 2; size <= npad; size <<= 1) {
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int t = threadIdx.x; t < npad / 2; t += kThreads) {
              const int lo = 2 * t - (t & (stride - 1)), hi = lo + stride;
              const unsigned long long a = key[lo], b = key[hi];
              if ((a > b) == ((lo & size) == 0)) {
                key[lo] = b;
                key[hi] = a;
              }
            }
          }
        }
        __syncthreads();
      }
      int4* list = reinterpret_cast<int4*>(smem + S::kList);
      for (int i = threadIdx.x; i < n_list; i += kThreads) {
        const int G = gridDim.x, c = blockIdx.x;
        const int k = i * G + ((i & 1) ? G - 1 - c : c);
        Unit w{};
        bool valid = false;
        if (k < total_units) {
          const int pk = k / per_s;
          valid = pair_unit<KVOWN>(p, sched, sorted ? (int)(unsigned)key[pk] : pk,
                                   k - pk * per_s, w);
        }
        list[3 * i] = make_int4(w.start, w.L, w.q0, w.g);
        list[3 * i + 1] = make_int4(w.h0, w.has1, w.kv_lo, w.n_kv);
        list[3 * i + 2] = make_int4(w.s, w.Lk, w.off, valid ? 1 : 0);
      }
      __syncthreads();
      sched.list = list;
      sched.n_list = n_list;
    } else {
      (void)n_list;
    }
  }
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  // Paged K/V: each producer warp keeps a window of its unit's page ids in registers,
  // lane i holding page base + i, plus the next 32 (loaded one block ahead), so that a
  // key tile's 8 ids come by shuffle instead of a dependent global load per tile.
  // Ids of pages past the sequence's end are -1; an out-of-range id is recorded and -1.
  auto page_id = [&](const Unit& w, int lp) -> int {
    if (!PAGED || lp * kPageRows >= w.Lk) return -1;  // decode_unit bounds Lk by max_pages
    int pid = p.page_table[(size_t)w.s * p.max_pages + lp];
    if (pid < 0 || pid >= p.num_pages) {
      atomicOr(p.err, kErrPageId);
      pid = -1;
    }
    return pid;
  };
  struct PageCursor {
    int base, cur, nxt;
  };
  auto cursor_start = [&](PageCursor& c, const Unit& w) {
    c.base = w.kv_lo * 8;
    c.cur = page_id(w, c.base + lane);
    c.nxt = page_id(w, c.base + 32 + lane);
  };
  // The 8 page ids of key tile `tile` (tiles are visited in increasing order) in pv[] of
  // every lane; bit i of the result is set when page i exists (whole warp calls).
  auto tile_pages = [&](PageCursor& c, const Unit& w, int tile, int (&pv)[8]) -> uint32_t {
    const int lp0 = tile * 8;
    if (lp0 >= c.base + 32) {  // tiles advance one at a time: at most one block step
      c.cur = c.nxt;
      c.base += 32;
      c.nxt = page_id(w, c.base + 32 + lane);
    }
    const int off = lp0 - c.base;
    uint32_t m = 0;
#pragma unroll
    for (int pi = 0; pi < 8; ++pi) {
      pv[pi] = __shfl_sync(0xffffffffu, c.cur, off + pi);
      m |= (pv[pi] >= 0 ? 1u : 0u) << pi;
    }
    return m;
  };
  // The TMA loads of a key tile into `dst` (K or V), contiguous (one elected lane) or
  // paged (the whole warp: lane 0 posts the byte count, lanes 0..7 each copy one 16-row
  // page block in the same instruction; a page block lands where its rows of a 128-row box
  // would, the 128-byte swizzle being periodic in 1024 bytes).
  // Row of the unit's first key in contiguous K/V (producers call it once per unit).
  auto key_row0 = [&](const Unit& w) -> int { return KVOWN ? p.cu_k[w.s] : w.start; };
  auto load_kv_tile = [&](uint32_t dst, const CUtensorMap* tm, uint32_t full, const Unit& w,
                          int j, const int (&pv)[8], uint32_t vmask, int krow0) {
    if constexpr (PAGED) {
      // whole warp: lane 0 posts the byte count, lanes 0..7 each copy their page
      if (lane == 0) mbar_arrive_expect_tx(full, __popc(vmask) * kPageRows * 128 * S::kBoxes);
      __syncwarp();
      int mine = pv[0];
#pragma unroll
      for (int pi = 1; pi < 8; ++pi) mine = (lane == pi) ? pv[pi] : mine;
      if (lane < 8 && ((vmask >> lane) & 1u)) {
#pragma unroll
        for (int bx = 0; bx < S::kBoxes; ++bx)
          tma_load_2d(dst + bx * S::kBoxBytes + lane * kPageRows * 128, tm, full, bx * 64,
                      (mine * p.Hkv + w.g) * kPageRows);
      }
    } else {
      (void)pv;
      (void)vmask;
      mbar_arrive_expect_tx(full, S::kTileBytes);
#pragma unroll
      for (int bx = 0; bx < S::kBoxes; ++bx)
        tma_load_3d(dst + bx * S::kBoxBytes, tm, full, bx * 64, w.g, krow0 + (w.kv_lo + j) * kBN);
    }
  };
  // Paged: rows of V stage `vstage` at or past the sequence's end (a partial last page, or
  // pages never loaded) may hold anything, even NaN; zero them so that p = 0 cannot meet a
  // non-finite v in the PV MMA. Whole warp; ends with the proxy fence.
  auto zero_v_tail = [&](uint32_t vstage, const Unit& w, int j) {
    if constexpr (PAGED) {
      const int rows_ok = w.Lk - (w.kv_lo + j) * kBN;
      if (rows_ok < kBN) {
        const int r0 = rows_ok < 0 ? 0 : rows_ok;
        const int chunks = (kBN - r0) * 8 * S::kBoxes;  // 16-byte chunks
        for (int c = lane; c < chunks; c += 32) {
          const int bx = c / ((kBN - r0) * 8), rem = c - bx * ((kBN - r0) * 8);
          const uint32_t a = vstage + bx * S::kBoxBytes + (r0 + rem / 8) * 128 + (rem & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
    } else {
      (void)vstage;
      (void)w;
      (void)j;
    }
  };
  static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * 168, "register split");

  if (warp < 4) {
    regs_dealloc<kRegsLow>();
    // head_dim 64: one producer for Q, K and V, one S issuer for both head tiles and one PV
    // issuer per tile. Paged K/V (sixteen 16-row page copies per step) use the head_dim-128
    // roles instead (Q and K from warp 0, V from warp 2, one S+PV issuer per tile): there a
    // single producer falls behind (chunked gpt-oss prefill 0.658 -> 0.619 ms), while the
    // contiguous calls are faster this way (causal 0.754 -> 0.744 ms).
    if constexpr (TmemCols<D>::kSepP && !PAGED) {
      using C = TmemCols<D>;
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
      constexpr uint32_t hi = sdesc_sw128_hi(1024);
      auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
      };
      if (warp == 0) {
        // ================ head_dim 64: TMA producer of Q, K and V ================
        static_assert(S::kBoxes == 1, "one 128-byte column block per row at head_dim 64");
        // One warp walks the schedule; per unit the Q stage, then per step the K and the
        // V tile. K(j) and V(j) are loaded together, several steps ahead of their use.
        if (elect_one()) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
          tma_prefetch_desc(&tm_v);
        }
        int kc = 0, vc = 0, qc = 0;
        bool ok = true;
        Unit w;
        for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
          const int qs = qc % S::kNQ;
          if (!(ok = wait(bar(S::kBarQEmpty + qs), ((qc / S::kNQ) & 1) ^ 1))) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(S::kBarQFull + qs), (1 + w.has1) * S::kTileBytes);
            for (int t = 0; t <= w.has1; ++t)
              tma_load_3d(q_smem + (2 * qs + t) * S::kTileBytes, &tm_q, bar(S::kBarQFull + qs), 0,
                          w.h0 + t, w.start + w.q0);
          }
          __syncwarp();
          ++qc;
          PageCursor pc{};
          if constexpr (PAGED) cursor_start(pc, w);
          const int krow0 = PAGED ? 0 : key_row0(w);
          for (int j = 0; j < w.n_kv; ++j) {
            const int ks = kc % S::kNK, vs = vc % S::kNV;
            int pv[8];
            uint32_t vmask = 0;
            if constexpr (PAGED) vmask = tile_pages(pc, w, w.kv_lo + j, pv);
            if (!(ok = wait(bar(S::kBarKEmpty + ks), ((kc / S::kNK) & 1) ^ 1))) break;
            if (PAGED || elect_one())
              load_kv_tile(k_smem + ks * S::kTileBytes, &tm_k, bar(S::kBarKFull + ks), w, j, pv, vmask, krow0);
            __syncwarp();
            ++kc;
            if (!(ok = wait(bar(S::kBarVEmpty + vs), ((vc / S::kNV) & 1) ^ 1))) break;
            if (PAGED || elect_one())
              load_kv_tile(v_smem + vs * S::kTileBytes, &tm_v, bar(S::kBarVFull + vs), w, j, pv, vmask, krow0);
            __syncwarp();
            ++vc;
          }
        }
        // Let every copy still in flight land before the CTA may exit.
        if (lane == 0) {
          for (int i = max(0, kc - S::kNK); i < kc; ++i)
            mbar_drain(bar(S::kBarKFull + i % S::kNK), (i / S::kNK) & 1, p.timeout_ns);
          for (int i = max(0, vc - S::kNV); i < vc; ++i)
            mbar_drain(bar(S::kBarVFull + i % S::kNV), (i / S::kNV) & 1, p.timeout_ns);
          for (int i = max(0, qc - S::kNQ); i < qc; ++i)
            mbar_drain(bar(S::kBarQFull + i % S::kNQ), (i / S::kNQ) & 1, p.timeout_ns);
        }
      } else if (warp == 1) {
        // ============== head_dim 64: S issuer for both head tiles ==============
        // S_t(j) = Q_t K_j^T once the softmax of tile t has read S_t(j-1); K stage j is
        // released after both tiles' S, the Q stage after the unit's last S.
        const uint32_t lo_q0 = sdesc_sw128_lo(q_smem, 16);
        const uint32_t lo_k0 = sdesc_sw128_lo(k_smem, 16);
        int kc = 0, qc = 0;
        int sf0 = 0, sf1 = 0;  // S issued so far per head tile (s_free phases)
        bool ok = true;
        Unit w;
        for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
          const int qs = qc % S::kNQ;
          if (!(ok = wait(bar(S::kBarQFull + qs), (qc / S::kNQ) & 1))) break;
          ++qc;
          for (int j = 0; ok && j < w.n_kv; ++j) {
            const int ks = kc % S::kNK;
            if (!(ok = wait(bar(S::kBarKFull + ks), (kc / S::kNK) & 1))) break;
            const uint32_t bk = lo_k0 + ks * (S::kTileBytes >> 4);
            for (int t = 0; t <= w.has1; ++t) {
              const int sf = t ? sf1 : sf0;
              if (sf > 0 && !(ok = wait(bar(S::kBarSFree + t), (sf - 1) & 1))) break;
              tc_fence_after_sync();
              const uint32_t aq = lo_q0 + (2 * qs + t) * (S::kTileBytes >> 4);
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = kk * 2;  // 32 bytes per K=16 step
                  umma_ss(tmem + C::s(t), sdesc_join(aq + off, hi), sdesc_join(bk + off, hi), idS,
                          kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(S::kBarSFull + t));
              }
              __syncwarp();
              if (t) ++sf1; else ++sf0;
            }
            if (!ok) break;
            if (elect_one()) {
              umma_commit(bar(S::kBarKEmpty + ks));
              if (j == w.n_kv - 1) umma_commit(bar(S::kBarQEmpty + qs));
            }
            __syncwarp();
            ++kc;
          }
        }
        if (elect_one()) {
          umma_commit(bar(S::kBarDrain + 2));
          mbar_drain(bar(S::kBarDrain + 2), 0, p.timeout_ns);
        }
        __syncwarp();
      } else {
        // ============= head_dim 64: PV issuer of head tile t (warps 2, 3) =============
        // O_t += P_t V_j once V_j is resident, O_t was read out (a unit's first step) and
        // the softmax has written P_t(j); the wait for P comes last so the MMAs follow it
        // directly. V stages are released by both PV issuers (count 2).
        const int t = warp - 2;
        const uint32_t lo_v0 = sdesc_sw128_lo(v_smem, S::kBoxBytes);
        int vc = 0, pf = 0, uc = 0;
        bool ok = true;
        Unit w;
        for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
          if (t == 1 && !w.has1) {  // this tile is absent: only keep the V ring in step
            vc += w.n_kv;
            continue;
          }
          const int nrel = (w.has1 || t == 1) ? 1 : 2;
          for (int jp = 0; jp < w.n_kv; ++jp) {
            const int vs = vc % S::kNV;
            if (!(ok = wait(bar(S::kBarVFull + vs), (vc / S::kNV) & 1))) break;
            if (jp == 0 && uc > 0 && !(ok = wait(bar(S::kBarOFree + t), (uc - 1) & 1))) break;
            if (!(ok = wait(bar(S::kBarPFull + t), pf & 1))) break;
            zero_v_tail(v_smem + vs * S::kTileBytes, w, jp);
            tc_fence_after_sync();
            const uint32_t bv = lo_v0 + vs * (S::kTileBytes >> 4);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                umma_ts(tmem + C::o(t), tmem + C::p(t) + kk * 8,
                        sdesc_join(bv + kk * (2048 >> 4), hi), idPV, (jp > 0 || kk > 0) ? 1u : 0u);
              umma_commit(bar(S::kBarODone + t));
              for (int r2 = 0; r2 < nrel; ++r2) umma_commit(bar(S::kBarVEmpty + vs));
            }
            __syncwarp();
            ++vc;
            ++pf;
          }
          ++uc;
        }
        if (elect_one()) {
          umma_commit(bar(S::kBarDrain + t));
          mbar_drain(bar(S::kBarDrain + t), 0, p.timeout_ns);
        }
        __syncwarp();
      }
    } else {
    if (warp == 0) {
    // ========================= TMA producer: Q and K =========================
    // Q and K are needed early (S_t(j+1) is issued while the softmax still works on
    // step j), V only after the softmax; separate producers keep K from waiting behind V.
    // The whole warp walks the schedule; one elected lane issues the copies.
    {
      if (elect_one()) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      }
      int kc = 0, qc = 0;
      bool ok = true;
      Unit w;
      for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
        const int qs = qc % S::kNQ;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarQEmpty + qs), ((qc / S::kNQ) & 1) ^ 1, wc));
        if (!ok) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(S::kBarQFull + qs), (1 + w.has1) * S::kTileBytes);
          for (int t = 0; t <= w.has1; ++t) {
#pragma unroll
            for (int bx = 0; bx < S::kBoxes; ++bx)
              tma_load_3d(q_smem + (2 * qs + t) * S::kTileBytes + bx * S::kBoxBytes, &tm_q,
                          bar(S::kBarQFull + qs), bx * 64, w.h0 + t, w.start + w.q0);
          }
        }
        __syncwarp();
        ++qc;
        PageCursor pc{};
        if constexpr (PAGED) cursor_start(pc, w);
        const int krow0 = PAGED ? 0 : key_row0(w);
        for (int j = 0; j < w.n_kv; ++j) {
          const int st = kc % S::kNK;
          int pv[8];
          uint32_t vmask = 0;
          if constexpr (PAGED) vmask = tile_pages(pc, w, w.kv_lo + j, pv);
          ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarKEmpty + st), ((kc / S::kNK) & 1) ^ 1, wc));
          if (!ok) break;
          if (PAGED || elect_one())
            load_kv_tile(k_smem + st * S::kTileBytes, &tm_k, bar(S::kBarKFull + st), w, j, pv, vmask, krow0);
          __syncwarp();
          ++kc;
        }
      }
      // Let every copy still in flight land before the CTA may exit.
      if (lane == 0) {
        for (int i = max(0, kc - S::kNK); i < kc; ++i)
          mbar_drain(bar(S::kBarKFull + i % S::kNK), (i / S::kNK) & 1, p.timeout_ns);
        for (int i = max(0, qc - S::kNQ); i < qc; ++i)
          mbar_drain(bar(S::kBarQFull + i % S::kNQ), (i / S::kNQ) & 1, p.timeout_ns);
      }
    }
    } else if (warp == 2) {
    // ============================ TMA producer: V ============================
    {
      if (elect_one()) tma_prefetch_desc(&tm_v);
      int vc = 0;
      bool ok = true;
      Unit w;
      for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
        PageCursor pc{};
        if constexpr (PAGED) cursor_start(pc, w);
        const int krow0 = PAGED ? 0 : key_row0(w);
        for (int j = 0; j < w.n_kv; ++j) {
          const int st = vc % S::kNV;
          int pv[8];
          uint32_t vmask = 0;
          if constexpr (PAGED) vmask = tile_pages(pc, w, w.kv_lo + j, pv);
          ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarVEmpty + st), ((vc / S::kNV) & 1) ^ 1, wc));
          if (!ok) break;
          if (PAGED || elect_one())
            load_kv_tile(v_smem + st * S::kTileBytes, &tm_v, bar(S::kBarVFull + st), w, j, pv, vmask, krow0);
          __syncwarp();
          ++vc;
        }
      }
      if (lane == 0) {
        for (int i = max(0, vc - S::kNV); i < vc; ++i)
          mbar_drain(bar(S::kBarVFull + i % S::kNV), (i / S::kNV) & 1, p.timeout_ns);
      }
    }
    } else if (warp == 1 || warp == 3) {
    // ======================== MMA issuers, one per head tile ========================
    // tcgen05.mma issue blocks while the tensor core is busy, so a single issuer for
    // both head tiles would make one tile's next S wait behind the other tile's PV.
    // Each tile has its own issuing thread (warp 1: tile 0, warp 3: tile 1) that follows
    // that tile's dependency order with blocking waits; the tensor core interleaves the
    // two queues. Shared K, V and Q stages are released by one commit from each issuer
    // (barrier count 2); for a unit with a single head tile, issuer 0 commits twice.
    // The whole warp walks the schedule and waits; one elected lane issues (issuing from
    // a converged warp keeps the descriptors warp-uniform, about twice as fast per MMA as
    // from a single-lane branch).
    {
      using C = TmemCols<D>;
      const int t = warp == 1 ? 0 : 1;
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
      // Shared-memory descriptors are built once; an MMA only adds a constant offset
      // (in 16-byte units) to the low half.
      constexpr uint32_t hi = sdesc_sw128_hi(1024);
      const uint32_t lo_q0 = sdesc_sw128_lo(q_smem, 16);
      const uint32_t lo_k0 = sdesc_sw128_lo(k_smem, 16);
      const uint32_t lo_v0 = sdesc_sw128_lo(v_smem, S::kBoxBytes);
      const uint32_t dS = tmem + C::s(t), dO = tmem + C::o(t), aP = tmem + C::p(t);
      int kc = 0, vc = 0, qc = 0;
      int gs = 0;  // softmax steps of this tile before the current unit (s_free index)
      int uc = 0;  // units this tile finished (o_free parity)
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
      };
      Unit w;
      for (int r = 0; ok && next_unit<KVOWN, LIST>(p, sched, r, w);) {
        const int n = w.n_kv;
        const int qs = qc % S::kNQ;
        const int nrel = (w.has1 || t == 1) ? 1 : 2;  // commits owed to shared stages
        if (t == 1 && !w.has1) {  // this tile is absent: only keep the ring counters in step
          ++qc;
          kc += n;
          vc += n;
          continue;
        }
        if (!(ok = wait(bar(S::kBarQFull + qs), (qc / S::kNQ) & 1))) break;
        ++qc;
        const uint32_t aq = lo_q0 + (2 * qs + t) * (S::kTileBytes >> 4);
        // S_t(j): K_j resident and S_t free (read by the softmax, or P_t(j-1) consumed).
        auto do_s = [&](int j) -> bool {
          const int ks = kc % S::kNK;
          if (!wait(bar(S::kBarKFull + ks), (kc / S::kNK) & 1)) return false;
          if (C::kSepP) {
            const int f = gs + j - 1;  // the softmax step that last read S_t
            if (f >= 0 && !wait(bar(S::kBarSFree + t), f & 1)) return false;
          }
          tc_fence_after_sync();
          const uint32_t bk = lo_k0 + ks * (S::kTileBytes >> 4);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              constexpr int kBox = S::kBoxBytes >> 4;
              const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 2;  // 32 bytes per K=16 step
              umma_ss(dS, sdesc_join(aq + off, hi), sdesc_join(bk + off, hi), idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(bar(S::kBarSFull + t));
            for (int r = 0; r < nrel; ++r) {
              umma_commit(bar(S::kBarKEmpty + ks));
              if (j == n - 1) umma_commit(bar(S::kBarQEmpty + qs));
            }
          }
          __syncwarp();
          ++kc;
          return true;
        };
        // PV_t(jp): P_t(jp) written, V_jp resident, O_t read out (first step of a unit).
        auto do_pv = [&](int jp) -> bool {
          const int vs = vc % S::kNV;
          // V and O are normally ready long before P: wait for them first, so that the
          // MMAs go out right after "P written" is seen.
          if (!wait(bar(S::kBarVFull + vs), (vc / S::kNV) & 1)) return false;
          if (jp == 0 && uc > 0 && !wait(bar(S::kBarOFree + t), (uc - 1) & 1)) return false;
          if (!wait(bar(S::kBarPFull + t), (gs + jp) & 1)) return false;
          zero_v_tail(v_smem + vs * S::kTileBytes, w, jp);
          tc_fence_after_sync();
          const uint32_t bv = lo_v0 + vs * (S::kTileBytes >> 4);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ts(dO, aP + kk * 8, sdesc_join(bv + kk * (2048 >> 4), hi), idPV,
                      (jp > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar(S::kBarODone + t));
            for (int r = 0; r < nrel; ++r) umma_commit(bar(S::kBarVEmpty + vs));
          }
          __syncwarp();
          ++vc;
          return true;
        };
        for (int j = 0; j <= n && ok; ++j) {
          if (C::kSepP) {
            // S_t(j+1) may run while the softmax still works on P_t(j).
            if (j < n && !(ok = do_s(j))) break;
            if (j >= 1 && !(ok = do_pv(j - 1))) break;
          } else {
            // P_t(j-1) overwrote S_t: PV_t(j-1) has to be issued before S_t(j).
            if (j >= 1 && !(ok = do_pv(j - 1))) break;
            if (j < n && !(ok = do_s(j))) break;
          }
        }
        gs += n;
        ++uc;
      }
      // Wait for every MMA this warp issued before TMEM can be released.
      if (elect_one()) {
        umma_commit(bar(S::kBarDrain + t));
        mbar_drain(bar(S::kBarDrain + t), 0, p.timeout_ns);
      }
      __syncwarp();
    }
    }
    }  // head_dim 128 roles
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
    using C = TmemCols<D>;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t ts = tl + C::s(t);
    const uint32_t tp = tl + C::p(t);
    const uint32_t to = tl + C::o(t);
    const float sl = p.scale_log2;
    const float2 sl2 = make_float2(sl, sl);
    int sc = 0, pv = 0;
    bool ok = true;
    const bool pp = p.pingpong != 0;
    if (pp && t == 1) named_barrier_arrive(kNbTurn + 0, 256);  // warpgroup 0 goes first
    // Position for the dry tail: current unit, step, and the step's turn operations done
    // (0 none, 1 turn taken, 2 turn handed over).
    int r = 0, j = 0, stage = 2;
    Unit w;
    w.n_kv = 0;
    // DEFER (windowed head_dim 64, whose units are two or three steps long): a unit's
    // epilogue runs inside this warpgroup's next unit, in its first step right after the P
    // store, so the wait for the unit's last PV overlaps that step's exponentials. The
    // pending row, 1/d and log-sum-exp wait in shared memory (the registers are all taken);
    // an epilogue is pending exactly when this warpgroup has finished a unit (pv > 0).
    // Measured: window 128 168 -> 150 us; the causal workload was slower this way.
    uint4* const pend = reinterpret_cast<uint4*>(smem + S::kPend) + (t * 128 + row);
    auto pending_epilogue = [&]() {
      const uint4 e = *pend;
      const int64_t orow = (int64_t)(((uint64_t)e.y << 32) | e.x);
      const float inv = __uint_as_float(e.z);
      const bool row_ok = orow >= 0;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (row_ok ? orow : 0) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t o[32];
        tmem_ld32(to + 32 * c4, o);
        uint32_t q4[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2)
          q4[e2] = pack_bf16x2(__uint_as_float(o[2 * e2]) * inv, __uint_as_float(o[2 * e2 + 1]) * inv);
        if (row_ok) {
          if (p.out32) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) st_global_v8(dst + c4 * 4 + 2 * e2, &q4[8 * e2]);
          } else {
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
              dst[c4 * 4 + e2] = make_uint4(q4[4 * e2], q4[4 * e2 + 1], q4[4 * e2 + 2], q4[4 * e2 + 3]);
          }
        }
      }
      if (p.lse && row_ok) p.lse[orow] = __uint_as_float(e.w);
      tc_fence_before_sync();
      mbar_arrive(bar(S::kBarOFree + t));
    };
    while (ok) {
      if (!next_unit<KVOWN, LIST>(p, sched, r, w)) {
        if constexpr (DEFER) {
          if (pv > 0) {  // the last unit's epilogue
            ok = __all_sync(0xffffffffu, mbar_wait(bar(S::kBarODone + t), (pv - 1) & 1, wc));
            if (ok) {
              tc_fence_after_sync();
              pending_epilogue();
            }
          }
        }
        break;
      }
      if (t == 1 && !w.has1) continue;
      const int h = w.h0 + t;
      const int i = w.q0 + row;  // query position inside its sequence
      float m = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
      float d = 1.f;  // the sink's own term exp2(sink - m) with m = sink
      for (j = 0; j < w.n_kv; ++j) {
        stage = 0;
        ok = mbar_wait(bar(S::kBarSFull + t), sc & 1, wc);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        ++sc;
        if (pp) named_barrier_sync(kNbTurn + t, 256);  // the other warpgroup's turn is over
        stage = 1;
        tc_fence_after_sync();
        const int k0 = (w.kv_lo + j) * kBN;
        const int pos0 = w.off + w.q0;  // key position of the tile's first query row
        const bool need_mask =
            (k0 + kBN - 1 > pos0) || (p.window > 0 && pos0 + kBM - 1 - k0 >= p.window);
        uint32_t r[kBN];
        // The row maximum comes with the load. A masked tile replaces it below with the
        // maximum of its visible columns; loading every tile the same way keeps one TMEM-load
        // form in the loop, which spares the softmax warps their register spills.
        float mx = tmem_ld128_max(ts, r);
        float s[kBN];
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(r[c]);
        if (C::kSepP) {  // S_t is in registers: the MMA may overwrite it with S_t(j+1)
          tc_fence_before_sync();
          mbar_arrive(bar(S::kBarSFree + t));
        }
        bool pv_done = (j == 0);  // PV_t(j-1) known complete
        if (need_mask) {
          // visible columns c: lo <= c <= hi
          const int hi = w.off + i - k0;
          const int lo = p.window > 0 ? w.off + i - k0 - p.window + 1 : INT_MIN;
          // One visibility word per 32 columns, then one bit test per column: fewer
          // instructions than two compares per column (gpt-oss causal 781 -> 761 us,
          // window 128 197 -> 167 us).
#pragma unroll
          for (int b = 0; b < kBN / 32; ++b) {
            const int hc = min(max(hi, 32 * b - 1), 32 * b + 31) - 32 * b;  // -1 .. 31
            const int lc = min(max(lo, 32 * b), 32 * b + 32) - 32 * b;      // 0 .. 32
            const uint32_t vis =
                hc >= lc ? (0xffffffffu >> (31 - hc)) & (0xffffffffu << lc) : 0u;  // bits lc..hc
#pragma unroll
            for (int c = 0; c < 32; ++c)
              s[32 * b + c] = (vis & (1u << c)) ? s[32 * b + c] : -INFINITY;
          }
          // Row maximum of the visible columns: 8 independent three-input chains, then 8 -> 1.
          float mp[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) mp[a] = fmax3(s[2 * a], s[2 * a + 1], s[16 + 2 * a]);
#pragma unroll
          for (int c = 32; c < kBN; c += 16) {
#pragma unroll
            for (int a = 0; a < 8; ++a) mp[a] = fmax3(mp[a], s[c + 2 * a], s[c + 2 * a + 1]);
          }
#pragma unroll
          for (int a = 0; a < 8; ++a) mp[a] = fmaxf(mp[a], s[17 + 2 * a]);
          mx = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
        }
        const float mnew = fmaxf(m, mx * sl);
        if (j == 0) {
          if (mnew > m) {
            d *= ex2(m - mnew);
            m = mnew;
          }
        } else if (__any_sync(0xffffffffu, mnew > m + kRescaleThreshold)) {
          // Some row's maximum moved far: the whole warp (TMEM access is warp-collective)
          // rescales its running outputs O to the new maxima; needs PV_{j-1} done.
          // Rescaling a row that did not need it is exact as well.
          const float alpha = (mnew == -INFINITY) ? 1.f : ex2(m - mnew);
          ok = mbar_wait(bar(S::kBarODone + t), (pv + j - 1) & 1, wc);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          tc_fence_after_sync();
#pragma unroll
          for (int c4 = 0; c4 < D / 16; ++c4) {
            uint32_t o[16];
            tmem_ld16(to + 16 * c4, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(to + 16 * c4, o);
          }
          tmem_st_wait();
          d *= alpha;
          m = mnew;
          pv_done = true;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        const float2 nmu = make_float2(-mu, -mu);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};  // independent partial row sums
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int e = 0; e < kBN / 2; ++e) {
          const float2 x = ffma2(make_float2(s[2 * e], s[2 * e + 1]), sl2, nmu);
          const float2 pe = make_float2(ex2(x.x), ex2(x.y));
          acc[e & 3] = fadd2(acc[e & 3], pe);
          pk[e] = pack_bf16x2(pe.x, pe.y);
        }
        if constexpr (D == 128) {
          // The turn ends after the exponentials: the arrive depends on the row sum, which
          // cannot be computed before the ex2 results.
          const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
          d += (a01.x + a23.x) + (a01.y + a23.y);
          if (pp) named_barrier_arrive_after(kNbTurn + (t ^ 1), 256, d);
        } else {
          // head_dim 64: no data dependency, so the compiler may hand the turn over while
          // exponentials are still in flight; measured faster than either explicit point
          // (after the S load, or before the exponentials) and than a strict turn.
          if (pp) named_barrier_arrive(kNbTurn + (t ^ 1), 256);
        }
        stage = 2;
        // DEFER, first step with an epilogue pending: the previous unit's last PV must have
        // read P_t before P_t(0) replaces it (its O is read out after the P store).
        const bool defer_now = DEFER && j == 0 && pv > 0;
        if (C::kSepP && (!pv_done || defer_now)) {
          // P_t(j) replaces P_t(j-1): PV_t(j-1) must have read it.
          ok = mbar_wait(bar(S::kBarODone + t), (pv + j - 1) & 1, wc);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          tc_fence_after_sync();
        }
#pragma unroll
        for (int c4 = 0; c4 < kBN / 32; ++c4) {
          uint32_t q16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) q16[e] = pk[16 * c4 + e];
          tmem_st16(tp + 16 * c4, q16);
        }
        if constexpr (D != 128) {
          const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
          d += (a01.x + a23.x) + (a01.y + a23.y);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(S::kBarPFull + t));
        if constexpr (DEFER) {
          if (defer_now) pending_epilogue();
        }
      }
      if (!ok) break;
      j = w.n_kv - 1;  // every step of this unit is complete
      if constexpr (DEFER) {
        const int64_t orow = (i < w.L) ? (int64_t)(w.start + i) * p.Hq + h : -1;
        const float inv = d > 0.f ? 1.f / d : 0.f;
        const float lse_v = (d > 0.f && m != -INFINITY) ? (m + log2f(d)) * kLn2 : -INFINITY;
        *pend = make_uint4((uint32_t)(uint64_t)orow, (uint32_t)((uint64_t)orow >> 32),
                           __float_as_uint(inv), __float_as_uint(lse_v));
        pv += w.n_kv;
        continue;
      }
      // ---- epilogue: O / d -> bf16, rows of this sequence only ----
      ok = mbar_wait(bar(S::kBarODone + t), (pv + w.n_kv - 1) & 1, wc);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      pv += w.n_kv;
      tc_fence_after_sync();
      const float inv = d > 0.f ? 1.f / d : 0.f;
      const bool row_ok = i < w.L;
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)(w.start + i) * p.Hq + h) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t o[32];
        tmem_ld32(to + 32 * c4, o);
        uint32_t q4[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          q4[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        if (row_ok) {
          if (p.out32) {  // whole 32-byte sectors: measured 3% faster at head_dim 128
#pragma unroll
            for (int e = 0; e < 2; ++e) st_global_v8(dst + c4 * 4 + 2 * e, &q4[8 * e]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[c4 * 4 + e] = make_uint4(q4[4 * e], q4[4 * e + 1], q4[4 * e + 2], q4[4 * e + 3]);
          }
        }
      }
      // State's log-sum-exp: m and d are in the scaled exp2 domain (d relative to m).
      if (p.lse && row_ok)
        p.lse[(size_t)(w.start + i) * p.Hq + h] =
            (d > 0.f && m != -INFINITY) ? (m + log2f(d)) * kLn2 : -INFINITY;
      tc_fence_before_sync();
      mbar_arrive(bar(S::kBarOFree + t));
    }
    if (!ok && pp) {
      // Dry tail: the remaining turn hand-overs of this warp's schedule, all blocking.
      while (true) {
        for (; j < w.n_kv; ++j, stage = 0) {
          if (stage < 1) named_barrier_sync(kNbTurn + t, 256);
          if (stage < 2) named_barrier_sync(kNbTurn + (t ^ 1), 256);
        }
        do {
          if (!next_unit<KVOWN, LIST>(p, sched, r, w)) goto dry_done;
        } while (t == 1 && !w.has1);
        j = 0;
        stage = 0;
      }
    dry_done:;
    }
    // Warpgroup 1's hand-overs lead warpgroup 0's turns by one: take the last.
    if (pp && t == 0) named_barrier_sync(kNbTurn + 0, 256);
    __syncwarp();
    tc_fence_before_sync();
    named_barrier_sync(kNbTeardown, kThreads);
  }
}

template <int D, bool PAGED, bool KVOWN, bool DEFER = false>
cudaError_t launch(const PrefillLaunch& a, const PrefillParams& p, cudaStream_t stream) {
  using S = PrefillSmem<D>;
  const int grid0 = p.total_units < a.num_sms ? p.total_units : a.num_sms;
  // The CTA's unit list fits in shared memory: the snake schedule is used and even the
  // bound of every (q tile, sequence) pair being valid leaves at most kMaxListUnits per CTA.
  const bool list = S::kMaxListUnits > 0 && p.snake &&
                    (p.total_units + grid0 - 1) / grid0 <= S::kMaxListUnits;
  auto kern = list ? prefill_kernel<D, PAGED, KVOWN, DEFER, true>
                   : prefill_kernel<D, PAGED, KVOWN, DEFER, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.total_units < a.num_sms ? p.total_units : a.num_sms;
  kern<<<grid, kThreads, S::kBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream) {
  if (a.band) return launch_prefill_band(a, stream);
  PrefillParams p{};
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
  p.npairs = (p.G + 1) / 2;
  p.window = a.window;
  p.n_qt = (a.max_seqlen + kBM - 1) / kBM;
  const long long total = (long long)p.n_qt * a.num_seqs * a.num_kv_heads * p.npairs;
  if (total <= 0) return cudaSuccess;
  p.total_units = (int)total;
  p.snake = (a.num_seqs <= kMaxSchedSeqs && p.n_qt <= kMaxSchedQTiles &&
             (long long)a.num_seqs * p.n_qt < 65536) ? 1 : 0;
  p.pingpong = (p.G % 2 == 0) ? 1 : 0;
  p.scale_log2 = a.scale * kLog2e;
  p.timeout_ns = a.timeout_ns;
  p.kv_lens = a.kv_lens;
  p.page_table = a.page_table;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.max_kv = a.max_kv;
  p.cu_k = a.kv_lens ? nullptr : a.cu_seqlens_k;
  p.Tk = a.total_k;
  if (a.kv_lens)
    return a.head_dim == 64 ? launch<64, true, false>(a, p, stream)
                            : launch<128, true, false>(a, p, stream);
  if (p.cu_k)
    return a.head_dim == 64 ? launch<64, false, true>(a, p, stream)
                            : launch<128, false, true>(a, p, stream);
  if (a.head_dim == 64)
    return a.window > 0 ? launch<64, false, false, true>(a, p, stream)
                        : launch<64, false, false>(a, p, stream);
  return launch<128, false, false>(a, p, stream);
}

}  // namespace sa
