// Fused observation-row RoPE, attention scoring and keep-set selection on the
// fifth-generation tensor cores (tcgen05, TMEM accumulators, TMA loads).
//
// BeaconKV reading notes:
//   §2.3, Q_obs equation: beacons are rotated to the eviction step t, recent
//         queries keep their own positions tau;
//   §2.1 eq. 4: w_{r,j} = exp(q_r.k_j/sqrt d) / sum_{l accessible} exp(q_r.k_l/sqrt d),
//         where a recent row at tau reaches the keys at positions <= tau;
//   §2.3 eq. 7: Score[j] = max over every query head of the group and every
//         observation row of w_{r,j};
//   §2.3 eq. 8: I_final = Sort(prefix + recent window + TopK(Score, k_sel)).
//
// Score[j] = exp(max_r (l_rj - lse_r)), lse_r the row's log-sum-exp (the max of
// the weights is the exp of the max of the log-weights). Per unit (sequence,
// layer, KV head) the K slice streams through shared memory twice: pass 1
// keeps an online (max, sum) per observation row, pass 2 recomputes the
// logits and takes each key's max of l - lse. The second read of the slice
// follows the first at once and is served from L2.
//
// Precision: the rotated observation rows are split into bf16 hi + lo parts
// (residual below 2^-17 relative); both parts multiply the bf16 keys on the
// tensor cores into one fp32 accumulator, so a logit's error stays far below
// the 2e-3 score tolerance even for large logits.
//
// Structure: one persistent CTA per SM walks the units; its warps specialise.
//   warp 0   TMA producer: two 128-row x 64-column SWIZZLE_128B boxes per
//            128-key tile into a ring of shared-memory stages;
//   warp 1   TMEM owner and single-thread MMA issuer:
//              pass 1  D[row][key] = Q . K_tile^T   (M = 128 rows, N = 128 keys)
//              pass 2  D[key][row] = K_tile . Q^T   (M = 128 keys, N = rows)
//            so each epilogue thread owns one TMEM lane (a row in pass 1, a
//            key in pass 2) and reduces along its own registers only;
//   warp 2   compacts K and V of a unit whose keep set is known, with bulk
//            copies through shared memory, while later units are scored
//            (without compaction: warms L2 with the next unit's rows);
//   warp 3   selects the keep set of a finished unit from its scores;
//   warps 4-11  epilogue, two warpgroups taking alternate TMEM buffers:
//            TMEM -> registers, online log-sum-exp in pass 1, max-pooling in
//            pass 2, scores to shared memory; between units they build the
//            next unit's rotated rows (the tensor cores wait for them).
// L2 policies: pass-1 loads keep their lines (evict_last) so that pass 2
// finds them in L2, and pass 2 walks the tiles in reverse, newest first: when
// a unit's tiles do not all stay in L2, the ones pass 1 read last are the ones
// still there. Every compaction copy marks its lines evict_first.
//
// Every cross-warp wait is a bounded wait on an mbarrier; on expiry the kernel
// latches BKV_ERR_TIMEOUT, every role stops at its next wait, outstanding
// copies are drained and the TMEM is freed before the CTA exits.
//
// Selection drops the D = L - budget lowest-scoring candidates among slots
// [prefix, L - recent); among equal scores the higher slot is dropped first,
// so the lower slot wins a tie. Scores are >= 0, so their fp32 bit patterns
// order like the values: each lane keeps a sorted list of its smallest
// (score bits, ~slot) keys, the warp extracts the D smallest from the list
// heads, and a ballot scan writes the kept (and dropped) slots in order.
#include <atomic>

#include "score_common.cuh"

namespace bkv {

namespace {

// Large drop counts (D > kThresholdFrom): the D-th smallest candidate score x is
// found by a binary search over the 32-bit patterns (scores >= 0 order like
// their patterns) between the smallest and the largest, each step counting
// over the warp the candidates whose pattern is <= the midpoint (a warp-wide
// add per step). Up to 2048 candidates the lane's share stays in registers
// (the selector warp has the kernel's register budget to itself); beyond, the
// counts read shared memory. Every candidate below x is dropped, and among
// those equal to x the highest slots fill the rest.
constexpr int kThresholdFrom = 32;
constexpr int kRegCands = 64;  // candidates per lane held in registers
// Scores are weights in [0, 1]; NaN or +inf comes only from a non-finite
// input (a +inf logit, for one, turns its row's log-sum-exp into NaN or -inf).
constexpr float kInf = __builtin_huge_valf();
__device__ bool threshold_drop(const float* sc, int c0, int c1, int D, uint32_t* dropped) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int j = c0 + lane; j < c1; j += 32) {
    const float v = sc[j];
    bad |= !(v < kInf);  // NaN or +inf
    mn = min(mn, __float_as_uint(v));
    mx = max(mx, __float_as_uint(v));
  }
  // smallest x with #(patterns <= x) >= D lies in [lo, hi]; every midpoint is
  // below hi, so padding patterns of 0xFFFFFFFF are never counted
  uint32_t lo = __reduce_min_sync(kFull, mn), hi = __reduce_max_sync(kFull, mx);
  if (c1 - c0 <= 32 * kRegCands) {
    uint32_t v[kRegCands];
#pragma unroll
    for (int k = 0; k < kRegCands; ++k) {
      const int j = c0 + lane + 32 * k;
      v[k] = j < c1 ? __float_as_uint(sc[j]) : 0xFFFFFFFFu;
    }
    while (lo < hi) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      int c = 0;
#pragma unroll
      for (int k = 0; k < kRegCands; ++k) c += v[k] <= mid ? 1 : 0;
      if (__reduce_add_sync(kFull, c) >= D)
        hi = mid;
      else
        lo = mid + 1;
    }
  } else {
    while (lo < hi) {
      const uint32_t mid = lo + ((hi - lo) >> 1);
      int c = 0;
      for (int j = c0 + lane; j < c1; j += 32) c += __float_as_uint(sc[j]) <= mid ? 1 : 0;
      if (__reduce_add_sync(kFull, c) >= D)
        hi = mid;
      else
        lo = mid + 1;
    }
  }
  const uint32_t prefix = lo;  // the D-th smallest pattern
  // drop every candidate below the threshold, then those equal to it still
  // needed, highest slots first
  int below = 0;
  for (int j = c0 + lane; j < c1; j += 32)
    if (__float_as_uint(sc[j]) < prefix) {
      atomicOr(&dropped[j >> 5], 1u << (j & 31));
      ++below;
    }
  int need = D - __reduce_add_sync(kFull, below);
  for (int top = c1 - 1; top >= c0 && need > 0; top -= 32) {
    const int j = top - lane;  // lane 0 takes the highest slot of the chunk
    const bool tie = j >= c0 && __float_as_uint(sc[j]) == prefix;
    const unsigned tb = __ballot_sync(kFull, tie);
    const int before = __popc(tb & ((1u << lane) - 1u));  // ties at higher slots in this chunk
    if (tie && before < need) atomicOr(&dropped[j >> 5], 1u << (j & 31));
    need -= __popc(tb);
  }
  return __any_sync(kFull, bad);
}

// Small drop counts: each lane's kList smallest keys, then D warp minima.
__device__ bool list_drop(const float* sc, int c0, int c1, int D, uint32_t* dropped) {
  const int lane = threadIdx.x & 31;
  u64 list[kList];
  bool bad = false;
  // the lane's kList smallest keys above `after`
  auto fill = [&](u64 after) {
#pragma unroll
    for (int i = 0; i < kList; ++i) list[i] = kNoKey;
    for (int j0 = c0 + lane; j0 < c1; j0 += 32 * 8) {
      u64 k[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + 32 * i;
        k[i] = kNoKey;
        if (j < c1) {
          const float v = sc[j];
          bad |= !(v < kInf);  // NaN or +inf
          const u64 key = ((u64)__float_as_uint(v) << 32) | (uint32_t)~j;
          if (key > after) k[i] = key;
        }
      }
      sort8(k);
      if (k[0] < list[kList - 1]) merge8(list, k);
    }
  };
  fill(0ull);  // no real key is 0: that needs slot 0xFFFFFFFF
  int used = 0;
  __syncwarp();
  for (int d = 0; d < D; ++d) {
    u64 m = list[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const u64 o = __shfl_xor_sync(kFull, m, off);
      m = o < m ? o : m;
    }
    const int slot = (int)(~(uint32_t)m);
    if (lane == 0) atomicOr(&dropped[slot >> 5], 1u << (slot & 31));
    if (list[0] == m) {  // this lane owned it: pop, rebuild when empty
#pragma unroll
      for (int i = 0; i < kList - 1; ++i) list[i] = list[i + 1];
      list[kList - 1] = kNoKey;
      if (++used == kList) {
        fill(m);
        used = 0;
      }
    }
  }
  return __any_sync(kFull, bad);
}

// Keep set of one unit from its scores sc[0, L). One warp. The D = L - budget
// dropped slots are the D smallest 64-bit keys (score bits << 32 | ~slot)
// among the candidates [prefix, L - recent): lower score first, and among
// equal scores the higher slot first, so the lower slot wins a tie (scores
// are >= 0, so their bit patterns order like the values). Each lane keeps the
// kList smallest keys of its own candidates, built without data-dependent
// branches: batches of 8 keys are sorted by Batcher's odd-even network and
// merged into the list by a bitonic half-cleaner. The warp then extracts the
// global minimum D times; a lane whose list runs dry rebuilds it from the
// keys above the last one it gave up. dropped[] is a bitmask over slots;
// drops[] receives the dropped slots ascending. out[] receives the kept
// slots ascending, or with order_free the layout of the order-free
// compaction. Returns BKV_OK, BKV_ERR_NONFINITE if a score was NaN or +inf, or
// BKV_ERR_INTERNAL if the dropped set is not exactly D distinct candidate
// slots; drops[] then holds the D highest candidates instead, so that
// everything downstream stays in bounds.
__device__ uint32_t select_keep(const float* sc, int L, int prefix, int recent, int budget, int32_t* out,
                                uint32_t* dropped, int* drops, bool order_free, uint32_t* status) {
  static_assert(kList == 8, "the list networks are written for 8 keys");
  const int lane = threadIdx.x & 31;
  const int c0 = prefix < L ? prefix : L;
  const int c1 = L - recent > c0 ? L - recent : c0;
  const int D = L - budget;
  for (int wd = lane; wd < (L + 31) / 32; wd += 32) dropped[wd] = 0u;
  __syncwarp();
  const bool bad = D > kThresholdFrom ? threshold_drop(sc, c0, c1, D, dropped) : list_drop(sc, c0, c1, D, dropped);
  __syncwarp();
  // dropped slots ascending: per-word counts, a warp prefix sum, then the bits
  const int words = (L + 31) / 32;
  int dbase = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t bits = w < words ? dropped[w] : 0u;
    const int c = __popc(bits);
    int x = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    int pos = dbase + x - c;
    while (bits) {
      if (pos < D) drops[pos] = w * 32 + __ffs(bits) - 1;
      ++pos;
      bits &= bits - 1;
    }
    dbase += __shfl_sync(kFull, x, 31);
  }
  __syncwarp();
  // consistency of the keep set: exactly D dropped slots (the kept ones then
  // number budget), all of them candidates, so the prefix and the recent
  // window stay kept
  const bool consistent = dbase == D && (D == 0 || (drops[0] >= c0 && drops[D - 1] < c1));
  if (!consistent) {
    __syncwarp();
    for (int wd = lane; wd < (L + 31) / 32; wd += 32) dropped[wd] = 0u;
    __syncwarp();
    for (int i = lane; i < D; i += 32) {
      drops[i] = c1 - D + i;
      atomicOr(&dropped[(c1 - D + i) >> 5], 1u << ((c1 - D + i) & 31));
    }
    __syncwarp();
  }
  if (!order_free) {
    // kept slots ascending: a kept slot s goes to out[s - (dropped slots below s)],
    // one word of the dropped-slot mask (32 slots, one per lane) per round
    int below = 0;  // dropped slots in the words before w
    for (int w = 0; w < words; ++w) {
      const uint32_t bits = dropped[w];
      const int s = w * 32 + lane;
      if (s < L && !((bits >> lane) & 1u)) {
        const int pos = s - below - __popc(bits & ((1u << lane) - 1u));
        if (BKV_IN_RANGE(pos >= 0 && pos < budget, status)) out[pos] = s;
      }
      below += __popc(bits);
    }
  } else {
    // layout of the order-free compaction: slots below the budget keep their
    // rows, except the holes (dropped, ascending), which receive the kept slots
    // at or above the budget (ascending)
    int h = 0;  // holes = dropped slots below the budget = drops[0, h)
    for (int r0 = 0; r0 < D; r0 += 32) h += __popc(__ballot_sync(kFull, r0 + lane < D && drops[r0 + lane] < budget));
    for (int j = lane; j < budget; j += 32)
      if (!((dropped[j >> 5] >> (j & 31)) & 1u)) out[j] = j;
    for (int k = lane; k < h; k += 32) {
      int x = budget + k;  // the k-th slot >= budget that is not dropped
      for (int r = h; r < D && drops[r] <= x; ++r) ++x;
      if (BKV_IN_RANGE(drops[k] >= 0 && drops[k] < budget && x < L, status)) out[drops[k]] = x;
    }
  }
  return !consistent ? (uint32_t)BKV_ERR_INTERNAL : bad ? (uint32_t)BKV_ERR_NONFINITE : (uint32_t)BKV_OK;
}

// Miscellaneous shared memory: control word [0, 64), dropped-slot bitmask
// [64, 1088) (L <= 8192), copier chunk descriptors [1536, 1664), the copier's
// own copy of the dropped-slot bitmask [1664, 2688) and its per-word prefix
// counts [2688, 3712).
constexpr int kMiscBytes = 3712;
constexpr int kChunkRows = 32;                   // rows per compaction chunk
constexpr int kChunkBytes = kChunkRows * kD * 2;  // 8 KB
constexpr int kPfChunks = 16;                     // L2 prefetch lead of the copier in windows (few chunk buffers only)
constexpr int kRoundChunks = 2;                   // slot-order windows per copier round (<= half the chunk buffers)

struct Layout {
  int Rtot, chunks;                    // observation rows of a unit, row chunks of <= 256
  int R, Rp16, mtiles, qrows, rows64;  // rows per chunk, to 16, M tiles, rows allocated, rows to 64
  int ntiles, Lp, stages, bufcols, cbufs, scbufs, D;
  size_t q_hi, q_lo, kst, cst, sc, lse, lim, part, rowinfo, drops, bars, misc, total;
};

// Shared-memory plan. The fixed part holds the observation rows (bf16 hi and
// lo), the per-row statistics and tables; the rest goes to K-tile stages,
// compaction chunks and score buffers, in the first arrangement that fits:
// two or more K stages always, eight / four / two 8 KB compaction chunks when
// compacting in slot order (three stages and four chunks first for units
// split into two row chunks, whose passes read K twice as often), two chunks
// (and more K stages) for the order-free compaction, which moves at most
// L - budget rows; two score buffers (one when nothing else fits).
__host__ __device__ inline Layout make_layout_chunks(int Rtot, int L, int nr, int budget, int compact, int chunks) {
  Layout s;
  s.Rtot = Rtot;
  s.chunks = chunks;
  const int R = (Rtot + s.chunks - 1) / s.chunks;
  s.R = R;
  s.Rp16 = (R + 15) & ~15;
  s.mtiles = R > 128 ? 2 : 1;
  s.qrows = s.Rp16 > 128 ? s.Rp16 : 128;  // a second M tile covers rows [Rp16 - 128, Rp16)
  s.rows64 = (s.Rp16 + 63) / 64 * 64 > s.qrows ? (s.Rp16 + 63) / 64 * 64 : s.qrows;  // pass-2 column chunks
  s.ntiles = (L + kTileKeys - 1) / kTileKeys;
  s.Lp = s.ntiles * kTileKeys;
  s.bufcols = (s.mtiles > 1 || s.Rp16 > 128) ? 256 : 128;
  s.D = L - budget;
  const size_t qbytes = ((size_t)s.qrows * 256 + 1023) / 1024 * 1024;  // two 128-byte slabs per row
  const size_t small = (size_t)s.rows64 * 4 * (1 + s.chunks) + (size_t)s.qrows * 16 +
                       (size_t)s.chunks * s.qrows * 8 + 2 * (size_t)s.D * 4 + 16 + 64 * 8 + kMiscBytes + 64;
  const size_t cap = 227 * 1024 - 1024;  // 1 KB kept for aligning the dynamic base
  const size_t scb = (size_t)s.Lp * 4;
  static const int plans[][3] = {{4, 0, 2}, {3, 0, 2}, {2, 0, 2}, {2, 0, 1}};          // no compaction
  static const int cplans[][3] = {{2, 8, 2}, {2, 4, 2}, {2, 2, 2}, {2, 2, 1}};         // compaction
  static const int splans[][3] = {{3, 4, 2}, {2, 8, 2}, {2, 4, 2}, {2, 2, 1}};         // split units
  static const int oplans[][3] = {{4, 2, 2}, {3, 2, 2}, {2, 2, 2}, {2, 2, 1}};         // order-free
  s.stages = 0;
  s.cbufs = 0;
  s.scbufs = 0;
  for (int i = 0; i < 4; ++i) {
    const int* pl = compact == 2 ? oplans[i] : compact ? (chunks == 2 && Rtot <= 256 ? splans[i] : cplans[i]) : plans[i];
    const size_t need = 2 * qbytes + (size_t)pl[0] * kTileBytes + (size_t)pl[1] * kChunkBytes + pl[2] * scb + small;
    if (need <= cap) {
      s.stages = pl[0];
      s.cbufs = pl[1];
      s.scbufs = pl[2];
      break;
    }
  }
  size_t off = 0;
  s.q_hi = off;
  off += qbytes;
  s.q_lo = off;
  off += qbytes;
  s.kst = off;  // 1024-aligned
  off += (size_t)s.stages * kTileBytes;
  s.cst = off;
  off += (size_t)s.cbufs * kChunkBytes;
  s.sc = off;
  off += (size_t)s.scbufs * scb;
  s.lse = off;
  off += (size_t)s.rows64 * 4;
  s.lim = off;  // [chunks][rows64]
  off += (size_t)s.chunks * s.rows64 * 4;
  s.part = off;
  off += (size_t)s.qrows * 16;
  s.rowinfo = off;  // [chunks][qrows]
  off += (size_t)s.chunks * s.qrows * 8;
  s.drops = off;
  off += 2 * (size_t)s.D * 4 + 16;
  s.bars = (off + 15) & ~(size_t)15;
  off = s.bars + 64 * 8;
  s.misc = off;  // 16-byte aligned: the copier keeps int4 chunk descriptors here
  off += kMiscBytes;
  s.total = off + 1024;
  return s;
}

// More than 256 rows run as equal chunks (the last one padded with masked
// zero rows): two TMEM buffers of two M tiles hold 256 rows. Between 129 and
// 256 rows one chunk fits, but its rows (bf16 hi + lo) can leave the slot-
// order compaction fewer than four 8 KB chunk buffers, and the copier, short
// of bytes in flight, becomes the bound (R = 224 at budgets >= 1024: two
// buffers). Such units are then scored in two chunks of half the rows: K is
// read twice as often, but the freed shared memory gives the copier eight
// buffers (measured on R1-Distill-Qwen-7B's shape, batch 128: budget 1024
// 5.72 -> 4.72 ms, budget 4096 20.3 -> 17.8 ms; at budget 256, with four
// buffers already, two chunks were slower).
__host__ __device__ inline Layout make_layout(int Rtot, int L, int nr, int budget, int compact) {
  const int chunks = (Rtot + 255) / 256 > 0 ? (Rtot + 255) / 256 : 1;
  const Layout one = make_layout_chunks(Rtot, L, nr, budget, compact, chunks);
  if (chunks == 1 && Rtot > 128 && compact == 1 && one.cbufs < 4) {
    const Layout two = make_layout_chunks(Rtot, L, nr, budget, compact, 2);
    if (two.stages >= 2 && two.cbufs > one.cbufs) return two;
  }
  return one;
}

}  // namespace

// kChunked: more than 256 observation rows, scored in row chunks; the
// single-chunk instance compiles without the chunk bookkeeping.
template <bool kChunked>
__global__ void __launch_bounds__(kThreads, 1) score_select_kernel(const __grid_constant__ ScoreParams P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_head = P.nb + P.nr;
  const Layout lay = make_layout(P.group * per_head, P.L, P.nr, P.budget, P.compact);
  const int R = lay.R, L = P.L, T = lay.ntiles, S = lay.stages;
  const int NC = kChunked ? lay.chunks : 1;  // row chunks

  unsigned char* q_hi = smem + lay.q_hi;
  unsigned char* q_lo = smem + lay.q_lo;
  unsigned char* kst = smem + lay.kst;
  float* sc = reinterpret_cast<float*>(smem + lay.sc);    // [scbufs][Lp]
  float* lse = reinterpret_cast<float*>(smem + lay.lse);  // [qrows], log2 units
  int* lim = reinterpret_cast<int*>(smem + lay.lim);      // [qrows], exclusive key bound per row
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* kfull = bars;        // [4]
  uint64_t* kempty = bars + 4;   // [4]
  uint64_t* tfull = bars + 8;    // [2]
  uint64_t* tempty = bars + 10;  // [2]
  uint64_t* qready = bars + 12;
  uint64_t* qfree = bars + 13;
  uint64_t* sready = bars + 14;  // [2]
  uint64_t* sfree = bars + 16;   // [2]
  uint64_t* cfull = bars + 20;   // [8] compaction chunks landed in shared memory
  uint64_t* dready = bars + 28;  // [2] a unit's drop list is ready
  uint64_t* dfree = bars + 30;   // [2] the copier is done with a drop list
  unsigned char* cst = smem + lay.cst;                       // [cbufs][8 KB] compaction chunks
  int* dlist = reinterpret_cast<int*>(smem + lay.drops);     // [2][D] dropped slots, ascending
  const int NSC = lay.scbufs;                                // score buffers (1 or 2)
  uint64_t* lsebar = bars + 18;
  uint64_t* lse2bar = bars + 19;
  float* pm = reinterpret_cast<float*>(smem + lay.part);  // [2][qrows] per-group running max
  float* pz = pm + 2 * lay.qrows;                         // [2][qrows] per-group running sum
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + lay.misc);
  uint32_t* dropbits = reinterpret_cast<uint32_t*>(smem + lay.misc + 64);  // [ceil(L/32)], <= 8192 slots
  int2* rowinfo = reinterpret_cast<int2*>(smem + lay.rowinfo);             // [R] source offset, table row

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiThreads);       // one group consumes each buffer
      mbar_init(&sready[i], 2 * kEpiThreads);
      mbar_init(&sfree[i], 32);
    }
    mbar_init(qready, 2 * kEpiThreads);  // the epilogue warps build the rows
    mbar_init(qfree, 1);
    for (int i = 0; i < lay.cbufs; ++i) mbar_init(&cfull[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dready[i], 32);
      mbar_init(&dfree[i], 1);
    }
    mbar_init(lsebar, 2 * kEpiThreads);
    mbar_init(lse2bar, 2 * kEpiThreads);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // zero both row buffers once: padding rows stay zero for the whole launch
  for (int i = tid; i < (int)(2 * (lay.q_lo - lay.q_hi) / 16); i += kThreads)
    reinterpret_cast<uint4*>(q_hi)[i] = make_uint4(0, 0, 0, 0);
  // per-launch tables, chunk by chunk: the key bound and the source of each row
  for (int c = 0; c < NC; ++c)
    fill_row_tables(lim + c * lay.rows64, rowinfo + c * lay.qrows, c * R, R, lay.Rtot, lay.rows64, lay.qrows,
                    P.nb, P.nr, L, P.fps_cap, P.n_rq, P.ring_first, tid, kThreads);
  const uint32_t ncols = 2 * (uint32_t)lay.bufcols;
  if (warp == 1) tmem_alloc(&ctl->tmem_base, ncols);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int mine = P.units > (int)blockIdx.x ? (P.units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  const float qk_scale = kLog2e * rsqrtf((float)kD);  // rows carry 1/sqrt(d) and log2(e)
  const uint32_t slab_q = (uint32_t)lay.qrows * 128;
  auto head_base = [&](int it) -> int64_t {
    int layer, seq, kvh;
    unit_geom(blockIdx.x + it * gridDim.x, P.batch, P.kv_heads, layer, seq, kvh);
    return ((int64_t)layer * P.batch + seq) * (P.kv_heads * P.group) + (int64_t)kvh * P.group;
  };
  // source of row r of chunk c (nullptr: zero padding)
  auto row_src = [&](int64_t head0, int c, int r) -> const uint4* {
    const int2 info = rowinfo[c * lay.qrows + r];
    if (info.x < 0) return nullptr;
    const uint4* base = (info.x & (1 << 30)) ? P.rq + head0 * P.n_rq * 16 : P.bq + head0 * P.fps_cap * 16;
    return base + (info.x & ~(1 << 30));
  };
  // rotated observation rows of chunk c of unit `it`; thread t of n
  auto build_rows = [&](int it, int c, int t, int n) {
    const int64_t head0 = head_base(it);
    build_obs_rows(q_hi, q_lo, slab_q, R, rowinfo + c * lay.qrows, P.bq + head0 * P.fps_cap * 16,
                   P.rq + head0 * P.n_rq * 16, P.rope, qk_scale, t, n);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(qready);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;     // tiles issued
      int st = 0;          // stage of tile g (g mod S)
      uint32_t kph = 0;    // parity of (g div S)
      bool ok = true;
      const uint64_t keep = policy_evict_last(), stream = policy_evict_normal();
      for (int it = 0; it < mine && ok; ++it) {
        int layer, seq, kvh;
        unit_geom(blockIdx.x + it * gridDim.x, P.batch, P.kv_heads, layer, seq, kvh);
        const int row0 = (seq * P.kv_heads + kvh) * P.max_cache;
        for (int s2 = 0; s2 < 2 * T * NC; ++s2) {
          const int s = s2 % (2 * T);  // each row chunk runs both passes
          if (g >= S && !mbar_wait(&kempty[st], kph ^ 1u, ctl, P.status)) {
            ok = false;
            break;
          }
          const int kt = s < T ? s : 2 * T - 1 - s;  // pass 2 walks the tiles backwards
          mbar_expect_tx(&kfull[st], kTileBytes);
          const uint32_t dst = smem_u32(kst + (size_t)st * kTileBytes);
          const uint64_t pol = s < T ? keep : stream;
          tma_load_2d(dst, &P.kmap[layer], 0, row0 + kt * kTileKeys, &kfull[st], pol);
          tma_load_2d(dst + kSlabBytes, &P.kmap[layer], 64, row0 + kt * kTileKeys, &kfull[st], pol);
          ++g;
          if (++st == S) {
            st = 0;
            kph ^= 1u;
          }
        }
      }
      // drain: every load issued has landed before the CTA may exit
      for (int st = 0; st < S && st < g; ++st) {
        const long long last = g - 1 - ((g - 1 - st) % S);
        const long long t0 = clock64();
        while (!mbar_test(&kfull[st], (uint32_t)((last / S) & 1)) && clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      long long g = 0;   // tiles consumed
      int st = 0;        // stage of tile g (g mod S)
      uint32_t kph = 0;  // parity of (g div S)
      bool ok = true;
      const uint32_t qh = smem_u32(q_hi), ql = smem_u32(q_lo);
      const uint32_t slab_q = (uint32_t)lay.qrows * 128;  // bytes of one 64-column slab of the rows
      const uint32_t id1 = idesc_bf16(128, 128), id2 = idesc_bf16(128, lay.Rp16);
      int ci = 0;  // row chunks started
      for (int it = 0; it < mine && ok; ++it) {
        for (int c = 0; c < NC && ok; ++c, ++ci) {
          ok = mbar_wait(qready, (uint32_t)(ci & 1), ctl, P.status);
          for (int s = 0; s < 2 * T && ok; ++s, ++g) {
            const int b = (int)(g & 1);
            ok = mbar_wait(&kfull[st], kph, ctl, P.status);
            if (ok && g >= 2) ok = mbar_wait(&tempty[b], (uint32_t)(((g >> 1) + 1) & 1), ctl, P.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kb = smem_u32(kst + (size_t)st * kTileBytes);
            const uint32_t d = tmem + (uint32_t)(b * lay.bufcols);
            if (s < T) {
              for (int mt = 0; mt < lay.mtiles; ++mt) {
  #pragma unroll
                for (int part = 0; part < 2; ++part) {
                  const uint32_t qbase = (part ? ql : qh) + (uint32_t)(mt ? lay.Rp16 - 128 : 0) * 128;
  #pragma unroll
                  for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk & 3) * 32;
                    const uint64_t a = sw128_desc(qbase + (uint32_t)(kk >> 2) * slab_q + off);
                    const uint64_t bd = sw128_desc(kb + (uint32_t)(kk >> 2) * kSlabBytes + off);
                    umma_bf16(d + (uint32_t)mt * 128, a, bd, id1, (part | kk) ? 1u : 0u);
                  }
                }
              }
            } else {
  #pragma unroll
              for (int part = 0; part < 2; ++part) {
                const uint32_t qbase = part ? ql : qh;
  #pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t off = (uint32_t)(kk & 3) * 32;
                  const uint64_t a = sw128_desc(kb + (uint32_t)(kk >> 2) * kSlabBytes + off);
                  const uint64_t bd = sw128_desc(qbase + (uint32_t)(kk >> 2) * slab_q + off);
                  umma_bf16(d, a, bd, id2, (part | kk) ? 1u : 0u);
                }
              }
            }
            umma_commit(&kempty[st]);
            umma_commit(&tfull[b]);
            if (++st == S) {
              st = 0;
              kph ^= 1u;
            }
          }
          if (ok) umma_commit(qfree);  // arrives when every MMA that read this chunk's rows is done
        }
      }
      // after an abort, let the MMAs already issued finish before the TMEM is freed
      if (!ok && g > 0) {
        const long long t0 = clock64();
        while (!mbar_test(&tfull[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1)) &&
               clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else if (warp == 2) {
    if (P.compact) {
      // ---------------------------------------------------------- in-place compaction
      // BeaconKV reading notes §2.3 eq. 8: K_hat = K[:, I_final], V_hat = V[:, I_final].
      // With the dropped slots d_0 < ... < d_{D-1}, the rows of run r,
      // (d_r, d_{r+1}), move down by r + 1 slots; rows below d_0 stay. Every
      // row's destination lies below its source, so when chunks are loaded in
      // increasing address order and each chunk is stored only after every
      // load up to its own has landed, a store overlaps only sources already
      // loaded, and every later load reads above every earlier store's
      // destination: loads may run ahead of stores.
      //
      // Long runs (L >= 64 D): one lane walks the runs in chunks of up to
      // kChunkRows rows, one bulk load and one bulk store per chunk, with up
      // to CB - 1 chunks loaded ahead; a chunk buffer is reloaded once the
      // store issued before the last one is done reading it. Its buffer and
      // phase counters wrap without division, since a 64-bit modulo per chunk
      // costs more than the copy issue itself.
      //
      // Short runs: the moved range (d_0, L) goes through shared memory in
      // windows of kChunkRows consecutive source rows at fixed offsets from
      // d_0 + 1 (one bulk load each, whatever runs they span); each run's part
      // of a window leaves with its own bulk store, the dropped rows skipped.
      // The whole warp issues: a round is up to RW windows, one per lane, and
      // the chunk buffers form S sets of RW, one set per round, with the loads
      // of the next S - 1 rounds in flight. Lane i always uses buffer i of a
      // set, so its own bulk groups tell when its buffer is free again. A
      // round's stores start once every load of the round has landed. A
      // window finds its runs and their shifts from the copier's own bitmask
      // of the unit's dropped slots and per-word prefix counts, with bit
      // operations instead of searches of the drop list.
      //
      // Order-free compaction: the k-th dropped slot below the budget (a hole)
      // receives the k-th kept slot at or above the budget. Sources and
      // destinations are disjoint, so rounds need no ordering. A round is one
      // window of 32 tail slots [budget + 32m, budget + 32m + 32): each lane
      // whose slot is kept copies its K and V rows into a set of two buffers
      // (K rows, V rows) and from there into its hole.
      {
        const int CB = lay.cbufs, D = lay.D;
        const bool ofree = P.compact == 2;
        const bool runs = !ofree && (long long)L >= 64LL * D;  // long runs: one lane, chunks along the runs
        const int RW = ofree ? 32 : (CB / 2 < kRoundChunks ? CB / 2 : kRoundChunks);  // chunks per round
        const int S = ofree ? CB / 2 : CB / RW;                                       // buffer sets
        uint32_t par = 0u;  // bit x: parity of the next completion of this lane's buffer in set x (order-free: the set's)
        int4* cdesc = reinterpret_cast<int4*>(smem + lay.misc + 1536);  // long runs: [cbufs] tensor, source row, rows, shift
        int lb = 0, sb = 0;  // long runs: next buffer to load into / to store from
        uint32_t sph = 0u;   // long runs: parity of buffer sb's next completion
        bool ok = true;
        const uint64_t stream = policy_evict_first();
        // number of dropped slots below x (dl ascending)
        auto drops_below = [&](const int* dl, int x) -> int {
          int lo = 0, hi = D;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (dl[mid] < x)
              lo = mid + 1;
            else
              hi = mid;
          }
          return lo;
        };
        for (int it = 0; it < mine && ok; ++it) {
          const int b = it & 1;
          ok = __all_sync(kFull, mbar_wait(&dready[b], (uint32_t)((it >> 1) & 1), ctl, P.status));
          if (!ok) break;
          const int* dl = dlist + b * D;
          int layer, seq, kvh;
          unit_geom(blockIdx.x + it * gridDim.x, P.batch, P.kv_heads, layer, seq, kvh);
          const size_t rowbase = (size_t)(seq * P.kv_heads + kvh) * P.max_cache;
          char* const tk = reinterpret_cast<char*>(P.Kc[layer] + rowbase * kD);
          char* const tv = reinterpret_cast<char*>(P.Vc[layer] + rowbase * kD);
          bulk_wait_read<0>();  // the previous unit's stores are done reading this lane's buffers
          __syncwarp();
          uint32_t inflight = 0u;  // bit x: this lane (order-free: the warp) has a load in flight in set x
          unsigned long long moved = 0;  // rows moved per tensor
          if (runs) {
            if (lane == 0) {
              const int first = D > 0 ? dl[0] + 1 : L;  // lowest source row that moves
              // chunk cursor over the runs of K, then of V: tensor ct, run cr, next source row crow
              int ct = 0, cr = 0, crow = first;
              auto next = [&](int4& c) -> bool {
                while (ct < 2 && D > 0) {
                  const int end = cr + 1 < D ? dl[cr + 1] : L;
                  if (crow < end) {
                    const int n = end - crow < kChunkRows ? end - crow : kChunkRows;
                    c = make_int4(ct, crow, n, cr + 1);  // run cr moves down by cr + 1 slots
                    crow += n;
                    // source rows inside the cache, destination rows inside the budget
                    if (!BKV_IN_RANGE(c.y > c.w && c.y + c.z <= L && c.y - c.w + c.z <= P.budget, P.status))
                      return false;
                    return true;
                  }
                  if (++cr < D) {
                    crow = dl[cr] + 1;
                  } else {
                    ++ct;
                    cr = 0;
                    crow = first;
                  }
                }
                return false;
              };
              // With few chunk buffers the loads alone keep too few bytes in
              // flight to cover HBM latency; the moved rows [first, L) of K,
              // then of V, are then prefetched into L2 kPfChunks windows ahead.
              const bool pf_on = CB <= 4;
              const int span = L - first;
              int pf_row = 0;  // rows prefetched so far, K's moved rows then V's
              auto prefetch_to = [&](int target) {
                target = target < 2 * span ? target : 2 * span;
                while (pf_row < target) {
                  const int pt = pf_row >= span ? 1 : 0;
                  const int off = pf_row - (pt ? span : 0);
                  int nr = span - off < kChunkRows ? span - off : kChunkRows;
                  nr = target - pf_row < nr ? target - pf_row : nr;
                  bulk_prefetch_l2((pt ? tv : tk) + (size_t)(first + off) * (kD * 2), (uint32_t)nr * (kD * 2));
                  pf_row += nr;
                }
              };
              if (pf_on) prefetch_to(kPfChunks * kChunkRows);
              auto load = [&](const int4 c) {
                cdesc[lb] = c;
                const uint32_t bytes = (uint32_t)c.z * (kD * 2);
                mbar_expect_tx(&cfull[lb], bytes);
                bulk_load(smem_u32(cst + (size_t)lb * kChunkBytes), (c.x ? tv : tk) + (size_t)c.y * (kD * 2), bytes,
                          &cfull[lb], stream);
                lb = lb + 1 == CB ? 0 : lb + 1;
                if (pf_on) prefetch_to((c.x ? span : 0) + c.y + c.z - first + kPfChunks * kChunkRows);
              };
              int pend = 0;
              int4 c;
              while (pend < CB - 1 && next(c)) {
                load(c);
                ++pend;
              }
              while (pend > 0) {
                ok = mbar_wait(&cfull[sb], sph, ctl, P.status);
                if (!ok) break;
                const int4 d = cdesc[sb];
                bulk_store((d.x ? tv : tk) + (size_t)(d.y - d.w) * (kD * 2), smem_u32(cst + (size_t)sb * kChunkBytes),
                           (uint32_t)d.z * (kD * 2), stream);
                bulk_commit();
                if (++sb == CB) {
                  sb = 0;
                  sph ^= 1u;
                }
                --pend;
                if (next(c)) {
                  bulk_wait_read<1>();  // the buffer reused now belonged to the store before the last one
                  load(c);
                  ++pend;
                }
              }
              if (!ok) {  // after an abort, loads already issued must land before the CTA exits
                for (; pend > 0; --pend) {
                  const long long t0 = clock64();
                  while (!mbar_test(&cfull[sb], sph) && clock64() - t0 < kWaitCycles) {
                  }
                  if (++sb == CB) {
                    sb = 0;
                    sph ^= 1u;
                  }
                }
              }
              moved = D > 0 ? (unsigned long long)(L - D - dl[0]) : 0ull;
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
          } else if (!ofree) {
            const int first = D > 0 ? dl[0] + 1 : L;  // lowest source row that moves
            // this unit's dropped slots as a bitmask with per-word prefix
            // counts, so that a window finds its runs with bit operations (the
            // selector's own mask already belongs to the next unit)
            uint32_t* cbits = reinterpret_cast<uint32_t*>(smem + lay.misc + 1664);  // [ceil(L/32)]
            int* cpre = reinterpret_cast<int*>(smem + lay.misc + 2688);             // drops in words < w
            const int words = (L + 31) / 32;
            for (int w = lane; w < words; w += 32) cbits[w] = 0u;
            __syncwarp();
            for (int i = lane; i < D; i += 32)
              if (BKV_IN_RANGE(dl[i] >= 0 && dl[i] < L, P.status)) atomicOr(&cbits[dl[i] >> 5], 1u << (dl[i] & 31));
            __syncwarp();
            for (int w0 = 0, base = 0; w0 < words; w0 += 32) {
              const int w = w0 + lane;
              const int c = w < words ? __popc(cbits[w]) : 0;
              int x = c;
#pragma unroll
              for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, x, off);
                if (lane >= off) x += y;
              }
              if (w < words) cpre[w] = base + x - c;
              base += __shfl_sync(kFull, x, 31);
            }
            __syncwarp();
            const int W = (L - first + kChunkRows - 1) / kChunkRows;  // windows per tensor
            const int nch = D > 0 ? 2 * W : 0;                        // K windows, then V windows
            const int nrounds = (nch + RW - 1) / RW;
            // With few chunk buffers the loads alone keep too few bytes in
            // flight to cover HBM latency; the windows kPfChunks ahead are then
            // prefetched into L2.
            const bool pf_on = CB <= 4;
            auto window = [&](int j, char*& src, int& s, int& n) {
              const bool v = j >= W;
              src = v ? tv : tk;
              s = first + (v ? j - W : j) * kChunkRows;
              n = L - s < kChunkRows ? L - s : kChunkRows;
            };
            if (pf_on && lane < kPfChunks && lane < nch) {
              char* src;
              int s0, n;
              window(lane, src, s0, n);
              bulk_prefetch_l2(src + (size_t)s0 * (kD * 2), (uint32_t)n * (kD * 2));
            }
            auto issue = [&](int g) {
              const int j = g * RW + lane, set = g % S;
              if (lane < RW && j < nch) {
                char* src;
                int s0, n;
                window(j, src, s0, n);
                const int bi = set * RW + lane;
                mbar_expect_tx(&cfull[bi], (uint32_t)n * (kD * 2));
                bulk_load(smem_u32(cst + (size_t)bi * kChunkBytes), src + (size_t)s0 * (kD * 2),
                          (uint32_t)n * (kD * 2), &cfull[bi], stream);
                inflight |= 1u << set;
                if (pf_on && j + kPfChunks < nch) {
                  window(j + kPfChunks, src, s0, n);
                  bulk_prefetch_l2(src + (size_t)s0 * (kD * 2), (uint32_t)n * (kD * 2));
                }
              }
            };
            for (int g = 0; g < S - 1 && g < nrounds; ++g) issue(g);
            for (int g = 0; g < nrounds; ++g) {
              const int j = g * RW + lane, set = g % S;
              const bool act = lane < RW && j < nch;
              if (S == 1) issue(g);  // a single set: its previous stores were drained below
              bool mok = true;
              if (act) {
                mok = mbar_wait(&cfull[set * RW + lane], (par >> set) & 1u, ctl, P.status);
                if (mok) {
                  par ^= 1u << set;
                  inflight &= ~(1u << set);
                }
              }
              ok = __all_sync(kFull, mok);
              if (!ok) break;
              if (act) {
                // the kept rows of window j, one bulk store per run
                char* dst;
                int s0, n;
                window(j, dst, s0, n);
                const uint32_t buf = smem_u32(cst + (size_t)(set * RW + lane) * kChunkBytes);
                // bit i of dm: slot s0 + i dropped; kept runs are the runs of
                // ones in keep, each moving down by the drops below its start
                const int w0 = s0 >> 5, sh = s0 & 31;
                const uint32_t lo = cbits[w0], hi = w0 + 1 < words ? cbits[w0 + 1] : 0u;
                const uint32_t dm = sh ? (lo >> sh) | (hi << (32 - sh)) : lo;
                const int r = cpre[w0] + __popc(lo & ((1u << sh) - 1u));  // drops below s0
                uint32_t keep = ~dm & (n < 32 ? (1u << n) - 1u : ~0u);
                while (keep) {
                  const int a = __ffs(keep) - 1;
                  const uint32_t gap = ~keep & (~0u << a);
                  const int b = gap ? __ffs(gap) - 1 : 32;
                  const int d0 = s0 + a - (r + __popc(dm & ((1u << a) - 1u)));
                  if (BKV_IN_RANGE(d0 >= 0 && d0 + (b - a) <= P.budget, P.status))
                    bulk_store(dst + (size_t)d0 * (kD * 2), buf + (uint32_t)a * (kD * 2), (uint32_t)(b - a) * (kD * 2),
                               stream);
                  keep = b < 32 ? keep & (~0u << b) : 0u;
                }
              }
              bulk_commit();
              if (S == 1) {
                bulk_wait_read<0>();
              } else if (g + S - 1 < nrounds) {
                bulk_wait_read<1>();  // round g - 1's stores are done reading the set reloaded now
                issue(g + S - 1);
              }
            }
            moved = D > 0 ? (unsigned long long)(L - D - dl[0]) : 0ull;
          } else {
            const int h = drops_below(dl, P.budget);  // holes
            const int nrounds = (L - P.budget + 31) / 32;
            // lane's tail slot in round m, whether it is kept, and its rank
            // among the kept tail slots (= the index of its hole)
            auto slot = [&](int m, int& x, int& rank) -> bool {
              x = P.budget + 32 * m + lane;
              if (x >= L) return false;
              const int below = drops_below(dl, x);
              rank = (x - P.budget) - (below - h);
              return !(below < D && dl[below] == x);
            };
            auto issue = [&](int m) {
              const int set = m % S;
              int x, rank;
              const bool kept = slot(m, x, rank);
              const unsigned bal = __ballot_sync(kFull, kept);
              if (!bal) return;
              const int row = __popc(bal & ((1u << lane) - 1u));
              if (lane == 0) {
                mbar_expect_tx(&cfull[2 * set], (uint32_t)__popc(bal) * (kD * 2));
                mbar_expect_tx(&cfull[2 * set + 1], (uint32_t)__popc(bal) * (kD * 2));
              }
              __syncwarp();
              if (kept) {
                bulk_load(smem_u32(cst + (size_t)(2 * set) * kChunkBytes + (size_t)row * (kD * 2)),
                          tk + (size_t)x * (kD * 2), kD * 2, &cfull[2 * set], stream);
                bulk_load(smem_u32(cst + (size_t)(2 * set + 1) * kChunkBytes + (size_t)row * (kD * 2)),
                          tv + (size_t)x * (kD * 2), kD * 2, &cfull[2 * set + 1], stream);
              }
              inflight |= 1u << set;
            };
            for (int m = 0; m < S - 1 && m < nrounds; ++m) issue(m);
            for (int m = 0; m < nrounds; ++m) {
              const int set = m % S;
              if (S == 1) issue(m);
              if (inflight & (1u << set)) {
                const bool w0 = mbar_wait(&cfull[2 * set], (par >> set) & 1u, ctl, P.status);
                ok = __all_sync(kFull, w0 && mbar_wait(&cfull[2 * set + 1], (par >> set) & 1u, ctl, P.status));
                if (!ok) break;
                par ^= 1u << set;
                inflight &= ~(1u << set);
                int x, rank;
                const bool kept = slot(m, x, rank);
                const int row = __popc(__ballot_sync(kFull, kept) & ((1u << lane) - 1u));
                if (kept && BKV_IN_RANGE(rank >= 0 && rank < h && dl[rank] < P.budget && x < L, P.status)) {
                  const int hole = dl[rank];
                  bulk_store(tk + (size_t)hole * (kD * 2),
                             smem_u32(cst + (size_t)(2 * set) * kChunkBytes + (size_t)row * (kD * 2)), kD * 2, stream);
                  bulk_store(tv + (size_t)hole * (kD * 2),
                             smem_u32(cst + (size_t)(2 * set + 1) * kChunkBytes + (size_t)row * (kD * 2)), kD * 2,
                             stream);
                }
              }
              bulk_commit();
              if (S == 1) {
                bulk_wait_read<0>();
              } else if (m + S - 1 < nrounds) {
                bulk_wait_read<1>();  // round m - 1's stores are done reading the set reloaded now
                issue(m + S - 1);
              }
            }
            moved = (unsigned long long)h;
          }
          if (!ok) {
            // after an abort, loads already issued must land before the CTA exits
            for (int set = 0; set < S; ++set) {
              if (!(inflight & (1u << set))) continue;
              const int n = ofree ? 2 : 1;
              for (int q = 0; q < n; ++q) {
                const int bi = ofree ? 2 * set + q : set * RW + lane;
                const long long t0 = clock64();
                while (!mbar_test(&cfull[bi], (par >> set) & 1u) && clock64() - t0 < kWaitCycles) {
                }
              }
            }
            break;
          }
          if (lane == 0) {
            if (moved && P.rows_moved) atomicAdd(P.rows_moved, moved);
            mbar_arrive(&dfree[b]);
          }
        }
        bulk_wait_all();  // every store has landed before the CTA may exit
      }
    } else {
      // ---------------------------------------------------------- L2 warmer
      // Pulls the next row chunk's source rows into L2 while the current one
      // is scored, so the row build at the chunk boundary reads from L2.
      const int nchunks = mine * NC;
      for (int ci = 0; ci + 1 < nchunks; ++ci) {
        const bool ok = __all_sync(kFull, mbar_wait(qready, (uint32_t)(ci & 1), ctl, P.status));
        if (!ok) break;
        const int64_t h1 = head_base((ci + 1) / NC);
        for (int r = lane; r < R; r += 32) {
          const char* src = reinterpret_cast<const char*>(row_src(h1, (ci + 1) % NC, r));
          if (!src) continue;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 128));
        }
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ keep-set selector
    for (int it = 0; it < mine; ++it) {
      const int b = it % NSC, db = it & 1;
      bool ok = __all_sync(kFull, mbar_wait(&sready[b], (uint32_t)((it / NSC) & 1), ctl, P.status));
      // the copier must be done with this drop-list buffer (unit it - 2)
      if (ok && P.compact && it >= 2)
        ok = __all_sync(kFull, mbar_wait(&dfree[db], (uint32_t)(((it >> 1) + 1) & 1), ctl, P.status));
      if (!ok) break;
      const int u = blockIdx.x + it * gridDim.x;
      const float* s_u = sc + (size_t)b * lay.Lp;
      const uint32_t code = select_keep(s_u, L, P.prefix, P.recent, P.budget, P.kept + (size_t)u * P.budget,
                                        dropbits, dlist + db * lay.D, P.compact == 2, P.status);
      if (code != BKV_OK && lane == 0) latch(P.status, code);
      if (P.scores) {
        float* so = P.scores + (size_t)u * P.max_cache;
        for (int j = lane; j < L; j += 32) so[j] = s_u[j];
      }
      __syncwarp();
      if (P.compact) mbar_arrive(&dready[db]);
      mbar_arrive(&sfree[b]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Two warpgroups alternate over the TMEM buffers: group e takes the tiles
    // with (global tile index & 1) == e. In pass 1 each keeps its own running
    // (max, sum) per row; the two are merged into lse at the end of pass 1.
    const int grp = (warp - 4) >> 2;
    const int et = tid - 128 - grp * kEpiThreads, q = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float neg_inf = __int_as_float(0xff800000u);
    const float inv_rows = 1.0f / (float)lay.Rtot;  // mean pooling
    const int C = NC;
    long long g = 0;
    bool ok = true;
    int ci = 0;                // row chunks done
    const int bt = tid - 128;  // 0..255 over both groups, for the row build
    if (mine > 0) build_rows(0, 0, bt, 2 * kEpiThreads);
    for (int it = 0; it < mine && ok; ++it) {
      const int b_sc = it % NSC;
      float* s_u = sc + (size_t)b_sc * lay.Lp;
      // Row chunks of a unit run one after another; chunk ch's rows have their
      // own lse, and the per-key pooled value is carried across chunks in s_u
      // (log2 of the max so far, or the sum so far) by the thread that owns the
      // key, which is the same thread in every chunk (2T tiles per chunk).
      for (int ch = 0; ch < C && ok; ++ch, ++ci) {
        const int* limc = lim + ch * lay.rows64;
        const int Rc = min(R, lay.Rtot - ch * R);  // real rows of this chunk
        const bool first = ch == 0, last = ch == C - 1;
        float run_m[2] = {neg_inf, neg_inf}, run_z[2] = {0.f, 0.f};
        for (int s = 0; s < 2 * T && ok; ++s, ++g) {
          const int b = (int)(g & 1);
          if (b == grp) {
            ok = __all_sync(kFull, mbar_wait(&tfull[b], (uint32_t)((g >> 1) & 1), ctl, P.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t col0 = tmem + lane_base + (uint32_t)(b * lay.bufcols);
            const int kt = s < T ? s : 2 * T - 1 - s;
            if (s < T) {
              // pass 1: this thread owns observation row et (and a row of the second M tile)
              for (int mt = 0; mt < lay.mtiles; ++mt) {
                const int row = mt ? lay.Rp16 - 128 + et : et;
                // The second M tile overlaps the first on rows below 128. tcgen05.ld
                // is warp-collective (.sync.aligned), so only whole warps may skip
                // it; lanes holding a duplicate row load and discard (bound 0
                // masks every key, which leaves their running max and sum as is).
                const bool dup = mt && row < 128;
                if (__all_sync(kFull, dup)) continue;
                const int bound = dup ? 0 : limc[row] - kt * kTileKeys;  // keys [0, bound) are visible
  #pragma unroll
                for (int h = 0; h < 4; h += 2) {
                  float v[64];
                  tmem_ld32(col0 + (uint32_t)(mt * 128 + h * 32), *reinterpret_cast<float(*)[32]>(&v[0]));
                  tmem_ld32(col0 + (uint32_t)(mt * 128 + h * 32 + 32), *reinterpret_cast<float(*)[32]>(&v[32]));
                  tmem_wait_ld();
                  if (bound < (h + 2) * 32) {
  #pragma unroll
                    for (int e = 0; e < 64; ++e)
                      if (h * 32 + e >= bound) v[e] = neg_inf;
                  }
                  float t0 = v[0], t1 = v[1], t2 = v[2], t3 = v[3];
  #pragma unroll
                  for (int e = 4; e < 64; e += 4) {
                    t0 = fmaxf(t0, v[e]);
                    t1 = fmaxf(t1, v[e + 1]);
                    t2 = fmaxf(t2, v[e + 2]);
                    t3 = fmaxf(t3, v[e + 3]);
                  }
                  const float nm = fmaxf(run_m[mt], fmaxf(fmaxf(t0, t1), fmaxf(t2, t3)));
                  if (nm != neg_inf) {
                    float z0 = run_m[mt] == neg_inf ? 0.f : run_z[mt] * fast_exp2(run_m[mt] - nm);
                    float z1 = 0.f, z2 = 0.f, z3 = 0.f;
  #pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                      z0 += fast_exp2(v[e] - nm);
                      z1 += fast_exp2(v[e + 1] - nm);
                      z2 += fast_exp2(v[e + 2] - nm);
                      z3 += fast_exp2(v[e + 3] - nm);
                    }
                    run_z[mt] = (z0 + z1) + (z2 + z3);
                    run_m[mt] = nm;
                  }
                }
              }
            } else {
              // pass 2: this thread owns key j of the tile; columns are observation rows
              const int j = kt * kTileKeys + et;
              const bool masked_tile = (kt + 1) * kTileKeys > L - P.nr + 1;
              if (P.pool_mean) {
                // mean pooling: the weights exp2(l - lse) summed over the rows
                // (inaccessible and padding rows add 0), divided by the row count
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                for (int c = 0; c < lay.Rp16; c += 64) {
                  float v[64];
                  tmem_ld32(col0 + (uint32_t)c, *reinterpret_cast<float(*)[32]>(&v[0]));
                  tmem_ld32(col0 + (uint32_t)c + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
                  tmem_wait_ld();
                  const float4* l4 = reinterpret_cast<const float4*>(lse + c);
                  if (!masked_tile && c + 64 <= Rc) {
  #pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                      const float4 l = l4[e >> 2];
                      a0 += fast_exp2(v[e] - l.x);
                      a1 += fast_exp2(v[e + 1] - l.y);
                      a2 += fast_exp2(v[e + 2] - l.z);
                      a3 += fast_exp2(v[e + 3] - l.w);
                    }
                  } else {
                    const int4* b4 = reinterpret_cast<const int4*>(limc + c);
  #pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                      const float4 l = l4[e >> 2];
                      const int4 bd = b4[e >> 2];
                      a0 += j < bd.x ? fast_exp2(v[e] - l.x) : 0.f;
                      a1 += j < bd.y ? fast_exp2(v[e + 1] - l.y) : 0.f;
                      a2 += j < bd.z ? fast_exp2(v[e + 2] - l.z) : 0.f;
                      a3 += j < bd.w ? fast_exp2(v[e + 3] - l.w) : 0.f;
                    }
                  }
                }
                if (j < L) {
                  const float a = ((a0 + a1) + (a2 + a3)) + (first ? 0.f : s_u[j]);
                  s_u[j] = last ? a * inv_rows : a;
                }
              } else {
                float m0 = neg_inf, m1 = neg_inf, m2 = neg_inf, m3 = neg_inf;
                for (int c = 0; c < lay.Rp16; c += 64) {
                  float v[64];
                  tmem_ld32(col0 + (uint32_t)c, *reinterpret_cast<float(*)[32]>(&v[0]));
                  tmem_ld32(col0 + (uint32_t)c + 32, *reinterpret_cast<float(*)[32]>(&v[32]));  // inside the buffer
                  tmem_wait_ld();
                  if (!masked_tile && c + 64 <= Rc) {
                    const float4* l4 = reinterpret_cast<const float4*>(lse + c);
    #pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                      const float4 l = l4[e >> 2];
                      m0 = fmaxf(m0, v[e] - l.x);
                      m1 = fmaxf(m1, v[e + 1] - l.y);
                      m2 = fmaxf(m2, v[e + 2] - l.z);
                      m3 = fmaxf(m3, v[e + 3] - l.w);
                    }
                  } else {
                    // padding rows carry lim = 0, so the visibility test masks them too
                    const float4* l4 = reinterpret_cast<const float4*>(lse + c);
                    const int4* b4 = reinterpret_cast<const int4*>(limc + c);
    #pragma unroll
                    for (int e = 0; e < 64; e += 4) {
                      const float4 l = l4[e >> 2];
                      const int4 bd = b4[e >> 2];
                      m0 = fmaxf(m0, j < bd.x ? v[e] - l.x : neg_inf);
                      m1 = fmaxf(m1, j < bd.y ? v[e + 1] - l.y : neg_inf);
                      m2 = fmaxf(m2, j < bd.z ? v[e + 2] - l.z : neg_inf);
                      m3 = fmaxf(m3, j < bd.w ? v[e + 3] - l.w : neg_inf);
                    }
                  }
                }
                float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                if (j < L) {
                  if (!first) mx = fmaxf(mx, s_u[j]);
                  // every key is visible to the newest observation row, so a
                  // log-weight of -inf on every row means a -inf logit: a
                  // non-finite key (+inf and NaN keys give NaN scores, which
                  // the selector reports)
                  if (last && mx == neg_inf) latch(P.status, BKV_ERR_NONFINITE);
                  s_u[j] = !last ? mx : (mx == neg_inf ? 0.f : fast_exp2(mx));
                }
              }
            }
            tc_fence_before();
            mbar_arrive(&tempty[b]);
          }
          if (s == T - 1) {
            // merge the two groups' row statistics into lse
            for (int mt = 0; mt < lay.mtiles; ++mt) {
              const int row = mt ? lay.Rp16 - 128 + et : et;
              if (mt && row < 128) continue;
              pm[grp * lay.qrows + row] = run_m[mt];
              pz[grp * lay.qrows + row] = run_z[mt];
            }
            mbar_arrive(lsebar);
            ok = __all_sync(kFull, mbar_wait(lsebar, (uint32_t)(ci & 1), ctl, P.status));
            if (!ok) break;
            if (grp == 0) {
              for (int mt = 0; mt < lay.mtiles; ++mt) {
                const int row = mt ? lay.Rp16 - 128 + et : et;
                if (mt && row < 128) continue;
                const float ma = pm[row], mb = pm[lay.qrows + row];
                const float mm = fmaxf(ma, mb);
                float zz = 0.f;
                if (mm != neg_inf)
                  zz = (ma == neg_inf ? 0.f : pz[row] * fast_exp2(ma - mm)) +
                       (mb == neg_inf ? 0.f : pz[lay.qrows + row] * fast_exp2(mb - mm));
                lse[row] = zz > 0.f ? mm + fast_log2(zz) : neg_inf;
              }
            }
            mbar_arrive(lse2bar);
            ok = __all_sync(kFull, mbar_wait(lse2bar, (uint32_t)(ci & 1), ctl, P.status));
            // this unit's scores go to sc[b_sc]: the selector must be done with unit it - NSC
            if (ok && first && it >= NSC)
              ok = __all_sync(kFull, mbar_wait(&sfree[b_sc], (uint32_t)(((it / NSC) + 1) & 1), ctl, P.status));
            if (!ok) break;
          }
          if (last && s == 2 * T - 1) mbar_arrive(&sready[b_sc]);
        }
        // rows of the next chunk: the MMAs of this one must be done with the buffers
        if (ok && (it + 1 < mine || !last)) {
          ok = __all_sync(kFull, mbar_wait(qfree, (uint32_t)(ci & 1), ctl, P.status));
          if (ok) build_rows(last ? it + 1 : it, last ? 0 : ch + 1, bt, 2 * kEpiThreads);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

size_t score_smem_bytes(int R, int L, int nr, int budget, int compact) {
  const Layout s = make_layout(R, L, nr, budget, compact);
  return s.stages >= 2 ? s.total : (size_t)1 << 30;  // no plan fits: not supported
}

namespace {

// Self-test of the bounded waits: four warps wait on an mbarrier that nothing
// arrives on; the first to run out latches BKV_ERR_TIMEOUT and raises the
// abort flag, which the others see at their next poll. Every thread exits.
__global__ void __launch_bounds__(128) wait_selftest_kernel(uint32_t* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ Ctl ctl;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    ctl.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0u, &ctl, status, limit);
  if (ok) latch(status, BKV_ERR_INTERNAL);  // nothing completes the phase
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* status, long long limit, cudaStream_t s) {
  wait_selftest_kernel<<<1, 128, 0, s>>>(status, limit);
  return cudaGetLastError();
}

bool encode_kmaps(ScoreParams& p, const void* const* K, int layers, int batch, int kv_heads,
                  int max_cache) {
  // the driver's encoder, looked up once per process (thread-safe static initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres) !=
            cudaSuccess ||
        qres != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode) return false;
  const cuuint64_t rows = (cuuint64_t)batch * kv_heads * max_cache;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTileKeys};
  const cuuint32_t estr[2] = {1, 1};
  for (int l = 0; l < layers; ++l) {
    const CUresult r = encode(&p.kmap[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(K[l]),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

cudaError_t launch_score_select(const ScoreParams& p, cudaStream_t s) {
  const int rows = p.group * (p.nb + p.nr);
  const size_t smem = score_smem_bytes(rows, p.L, p.nr, p.budget, p.compact);
  const bool chunked = make_layout(rows, p.L, p.nr, p.budget, p.compact).chunks > 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // the largest plan once per device and instance (one bit each); every launch then fits
  static std::atomic<unsigned long long> configured[2] = {{0}, {0}};
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (!(configured[chunked].load() & bit)) {
    e = chunked ? cudaFuncSetAttribute(score_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)
                : cudaFuncSetAttribute(score_select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured[chunked].fetch_or(bit);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = p.units < sms ? p.units : sms;  // one persistent CTA per SM
  if (chunked)
    score_select_kernel<true><<<grid, kThreads, smem, s>>>(p);
  else
    score_select_kernel<false><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
