// Block-level building blocks of the per-segment selection:
//   * radix digit selection (most significant digit first, with early stop)
//     over a candidate list held in shared memory,
//   * the composite selection that resolves boundary ties by source index,
//   * compaction of the selected entries at positions from warp ballots and a
//     block prefix scan, and
//   * a bitonic sort of the selected items for sorted output.
//
// The list is a structure of arrays in shared memory: raw key bits and the
// segment-local source index of every entry, in no particular order.
#pragma once

#include <cstddef>

#include "common.cuh"

namespace segtopk {

constexpr int kDigitBits = 8;
constexpr int kBuckets = 1 << kDigitBits;

// Per-pass scratch of the digit selection. Passes are counted over every
// selection a block makes: pass j uses slot j % 3 and clears slot (j+1) % 3,
// whose last readers finished before the barrier of pass j-1. So a pass
// needs one barrier, and consecutive selections need none between them. The
// compaction after a selection uses the slot of its last pass (kept, kmax),
// which the second pass of the next selection clears.
struct __align__(16) PassSlot {
  uint32_t hist[kBuckets]; // digit histogram (read with 16-byte loads)
  uint32_t and_w[2];       // AND / OR of the keys seen (one or two words)
  uint32_t or_w[2];
  uint32_t ncand;          // candidates stored in the position buffer
  uint32_t kept;           // compaction: entries written so far
  uint32_t nfin;           // counting finish: keys staged
  uint32_t ties;           // compaction: boundary entries taken by arrival so far
  unsigned long long kmax; // compaction: largest rank written
};

// Keys a warp gathers for the counting finish of a selection.
constexpr uint32_t kFinishMax = 64;

// Counters of the statistics build (per CTA, summed over the launch).
enum StatIndex : int {
  kStatCtas = 0,        // CTAs that served a segment slice
  kStatCycles = 1,      // clock cycles from start to exit
  kStatFirstBound = 2,  // cycles spent setting the first bound (sample or exact selection)
  kStatStream = 3,      // cycles of the stream (first bound included)
  kStatFinal = 4,       // cycles after the stream: final selection, merge, sort, output
  kStatChunks = 5,      // ring chunks streamed
  kStatTrims = 6,       // list trims during the stream
  kStatRestreams = 7,   // slices read a second time (speculative bound too tight)
  kStatListEntries = 8, // candidate-list entries at the end of the stream
  kStatSpec = 9,        // slices whose first bound came from a sample
  kStatDigitPasses = 10,// digit-selection passes (histogram passes) in the CTA
  kStatWaitCycles = 11, // cycles thread 0 spent waiting for copies
  kStatKeys = 12,       // keys of the slices
  kStatSlowChunks = 13, // chunk shares of warp 0 that held candidates
  kStatFallbackChunks = 14, // chunk offers that overflowed the list
  kStatSpecWarp = 15,   // small speculative selection: cycles of the per-warp minimums
  kStatSpecMerge = 16,  // ... of the merge of the warps' lists
  kStatSpecKeep = 17,   // ... of writing the kept sample keys
  kStatFinalSelect = 18,// cycles of a lone CTA's final selection (list to k entries)
  kStatFinalWrite = 19, // cycles of its output (sort and write)
  kStatSelPasses = 20,  // cycles of digit passes of every block selection
  kStatSelFinish = 21,  // cycles of their counting finishes
  kStatSelCompact = 22, // cycles of compactions of selected entries
  kStatCount = 24
};

// Adds to a per-CTA counter of the statistics build (thread 0; `ctl` is the
// CTA's control block); nothing in an ordinary build.
#ifdef SEGTOPK_STATS
#define SEGTOPK_STAT_ADD(i, v)                                                                     \
  do {                                                                                             \
    if (threadIdx.x == 0)                                                                          \
      ctl.stat[(i)] += (unsigned long long)(v);                                                    \
  } while (0)
#else
#define SEGTOPK_STAT_ADD(i, v)                                                                     \
  do {                                                                                             \
  } while (0)
#endif

// Control block at the start of dynamic shared memory. Every CTA of a cluster
// has the same layout, so a field can be addressed in a peer through DSMEM.
struct Ctrl {
  uint64_t bars[8];                  // one mbarrier per ring stage
  uint64_t scan_tot[2][32];          // per-warp packed totals of the block scans (double buffered)
  uint64_t red[32];                  // block reductions
  PassSlot slot[3];                  // digit selection passes (see PassSlot)
  uint64_t fin[kFinishMax];          // staging of the counting finish
  uint32_t hist_m0[kBuckets];        // cluster histogram merge: this CTA's histogram
  uint32_t hist_merged[kBuckets];    // cluster leader: histogram pushed by the other CTAs
  uint32_t res[4];                   // cluster leader: result of a merged pass
  uint32_t chunk_count[3];           // entries appended during a chunk (three in rotation)
  uint32_t gather_count;             // cluster leader: entries gathered from the cluster
  uint32_t front_base;               // cross-CTA scan: selected entries of preceding CTAs
  uint32_t tie_base;                 // cross-CTA scan: boundary ties of preceding CTAs
  uint32_t spec_kept;                // small speculative selection: sample keys kept
  uint64_t xb[16][2];                // cluster leader: every CTA's local k-th (rank, preference index)
  uint64_t xb_min[2];                // the cluster-wide minimum of xb
  uint32_t abort;                    // a wait on a bulk copy gave up: the CTA writes no output
  uint32_t pad_;
  unsigned long long stat[kStatCount]; // per-CTA counters of the statistics build
};
static_assert(sizeof(PassSlot) % 16 == 0, "every slot's histogram is 16-byte aligned");
static_assert(offsetof(Ctrl, slot) % 16 == 0, "the slots are 16-byte aligned");
static_assert(offsetof(PassSlot, kmax) % 8 == 0, "64-bit shared atomics need 8-byte alignment");
constexpr uint32_t kCtrlBytes = (sizeof(Ctrl) + 127u) & ~127u;

// Entries a selection reads: `count` list entries, then `ext_count` keys of
// a ring stage whose source indices are ext_idx0, ext_idx0 + 1, ...
template <class Raw>
struct Src {
  const Raw* raw;
  const uint32_t* idx;
  uint32_t count;
  const Raw* ext_raw;
  uint32_t ext_idx0;
  uint32_t ext_count;
  __device__ __forceinline__ uint32_t size() const { return count + ext_count; }
  __device__ __forceinline__ Raw key(uint32_t e) const { return e < count ? raw[e] : ext_raw[e - count]; }
  __device__ __forceinline__ uint32_t index(uint32_t e) const { return e < count ? idx[e] : ext_idx0 + (e - count); }
};

template <class Raw>
__device__ __forceinline__ Src<Raw> list_src(const Raw* raw, const uint32_t* idx, uint32_t count)
{
  return Src<Raw>{raw, idx, count, nullptr, 0u, 0u};
}

// Warp 0 of the block: find the bucket holding the krem-th best candidate.
// `h` holds the 8 bucket counts this lane owns (buckets 8*lane .. 8*lane+7).
// Writes bucket, count before it and its count to res[].
__device__ __forceinline__ void find_bucket(const uint32_t (&h)[8], uint32_t krem, uint32_t* res)
{
  const uint32_t lane = lane_id();
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    s += h[i];
  const uint32_t incl = warp_inclusive_sum(s);
  const uint32_t hit = __ballot_sync(kFull, incl >= krem);
  const uint32_t src = __ffs(hit) - 1; // the candidate total is always >= krem
  if (lane == src) {
    uint32_t before = incl - s;
    uint32_t b = 8 * lane + 7, cnt = h[7];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (before + h[i] >= krem) {
        b = 8 * lane + i;
        cnt = h[i];
        break;
      }
      before += h[i];
    }
    res[0] = b;
    res[1] = before;
    res[2] = cnt;
  }
}

// Every lane of the calling warp: the bucket of `hist` (16-byte aligned)
// holding the krem-th best candidate, the count before it and its count.
__device__ __forceinline__ void find_bucket_warp(const uint32_t* hist, uint32_t krem, uint32_t& b, uint32_t& before,
                                                 uint32_t& cnt)
{
  const uint32_t lane = lane_id();
  const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 2 * lane;
  const uint4 x = h4[0], y = h4[1];
  const uint32_t h[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  const uint32_t sum = (h[0] + h[1]) + (h[2] + h[3]) + (h[4] + h[5]) + (h[6] + h[7]);
  const uint32_t incl = warp_inclusive_sum(sum);
  const uint32_t src = __ffs(__ballot_sync(kFull, incl >= krem)) - 1; // the candidate total is always >= krem
  // within the source lane: the first of its buckets that reaches krem
  uint32_t cum = incl - sum, bb = 7, bf = 0, bc = 0;
  bool got = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hit = !got && cum + h[i] >= krem;
    bb = hit ? (uint32_t)i : bb;
    bf = hit ? cum : bf;
    bc = hit ? h[i] : bc;
    got |= hit;
    cum += h[i];
  }
  b = 8 * src + __shfl_sync(kFull, bb, src);
  before = __shfl_sync(kFull, bf, src);
  cnt = __shfl_sync(kFull, bc, src);
}

template <class Key>
struct Radix {
  Key prefix;      // resolved leading digits of the boundary key
  Key mask;        // which digits are resolved
  uint32_t krem;   // how many boundary candidates are still needed
  uint32_t cnt;    // candidates in the boundary bucket
  bool stopped;    // the whole boundary bucket may be taken (cnt - krem <= slack)
};

// Candidate-position buffer (shared memory) that a selection may use to
// visit only the boundary candidates after its first two passes.
struct CandBuf {
  uint16_t* pos;  // entry positions (an entry domain is < 65536 entries)
  uint32_t cap;
  uint32_t n;     // filled by radix_select: candidates stored, or ~0u if not compacted
};

// Folds a thread's AND / OR of keys into the shared words (one warp
// reduction and one native 32-bit atomic per word and warp).
__device__ __forceinline__ void fold_and_or(uint32_t* a, uint32_t* o, uint32_t va, uint32_t vo)
{
  va = __reduce_and_sync(kFull, va);
  vo = __reduce_or_sync(kFull, vo);
  if (lane_id() == 0) {
    atomicAnd(a, va);
    atomicOr(o, vo);
  }
}
__device__ __forceinline__ void fold_and_or(uint32_t* a, uint32_t* o, uint64_t va, uint64_t vo)
{
  fold_and_or(a, o, (uint32_t)va, (uint32_t)vo);
  fold_and_or(a + 1, o + 1, (uint32_t)(va >> 32), (uint32_t)(vo >> 32));
}
template <class Key>
__device__ __forceinline__ Key read_word(const uint32_t* w)
{
  if constexpr (sizeof(Key) == 8)
    return ((Key)w[1] << 32) | w[0];
  else
    return (Key)w[0];
}

// Clears a pass slot (block-wide part: histogram words by thread index).
template <int NT>
__device__ __forceinline__ void clear_slot(PassSlot& sl)
{
  for (uint32_t i = threadIdx.x; i < (uint32_t)kBuckets; i += NT)
    sl.hist[i] = 0;
  if (threadIdx.x == 0) {
    sl.and_w[0] = sl.and_w[1] = ~0u;
    sl.or_w[0] = sl.or_w[1] = 0u;
    sl.ncand = 0;
    sl.kept = 0;
    sl.nfin = 0;
    sl.ties = 0;
    sl.kmax = 0;
  }
}

// Counting finish of a selection, block-wide: the candidates (positions
// pos[0..npos)) whose key matches prefix under mask -- at most kFinishMax of
// them -- are staged in shared memory (counter *nfin, zero on entry); after
// one barrier every warp finds, by counting over registers and shuffles, the
// krem-th best key value v among them, the number of staged keys better
// than v and the number equal to it.
template <class Key, int NT, class Get>
__device__ __forceinline__ void finish_by_count(Key* stage, uint32_t* nfin, const uint16_t* pos, uint32_t npos,
                                                Key prefix, Key mask, uint32_t krem, Get&& get, Key& v, uint32_t& less,
                                                uint32_t& eq)
{
  for (uint32_t i = threadIdx.x; i < npos; i += NT) {
    Key key = 0;
    if (get((uint32_t)pos[i], key) && (key & mask) == prefix) {
      const uint32_t slot = atomicAdd(nfin, 1u);
      if (slot < kFinishMax)
        stage[slot] = key;
    }
  }
  __syncthreads();
  uint32_t n = *nfin;
  if (n > kFinishMax)
    n = kFinishMax; // cannot happen: the caller checked the bucket count
  const uint32_t lane = lane_id();
  const Key a = lane < n ? stage[lane] : (Key)0;
  const Key c = lane + 32 < n ? stage[lane + 32] : (Key)0;
  uint32_t la = 0, ea = 0, lc = 0, ec = 0;
  // staged keys j < n only (often a handful): the first 32 by one shuffle
  // each, keys 32..63 by a second one only when there are that many
  const uint32_t n0 = n < 32 ? n : 32u;
#pragma unroll 4
  for (uint32_t j = 0; j < n0; ++j) {
    const Key w0 = __shfl_sync(kFull, a, j);
    la += w0 < a;
    ea += w0 == a;
    lc += w0 < c;
    ec += w0 == c;
  }
  for (uint32_t j = 32; j < n; ++j) {
    const Key w1 = __shfl_sync(kFull, c, j - 32);
    la += w1 < a;
    ea += w1 == a;
    lc += w1 < c;
    ec += w1 == c;
  }
  const bool fa = lane < n && la < krem && krem <= la + ea;
  const bool fc = lane + 32 < n && lc < krem && krem <= lc + ec;
  const uint32_t bal = __ballot_sync(kFull, fa || fc);
  const uint32_t src = bal ? __ffs(bal) - 1 : 0u;
  const Key mine = fa ? a : c;
  const uint32_t ml = fa ? la : lc, me = fa ? ea : ec;
  v = __shfl_sync(kFull, mine, src);
  less = __shfl_sync(kFull, ml, src);
  eq = __shfl_sync(kFull, me, src);
}

// One radix selection: among the candidates (get(e, key) returns true) of
// the entries e of a domain -- [0, count), or the positions dom[0..dom_n) if
// dom is given -- find the kk best by key (smaller = better). Each pass
// histograms one 8-bit digit of the candidates whose resolved digits match,
// finds the bucket holding the krem-th best, narrows krem and folds the digit
// into the prefix; it stops when that bucket holds exactly krem candidates
// ("Implement Segmented TopK using Thread-Block-Clusters", sections 1.2
// "Radix (digit) top-k" and 1.4 "Early stop"). With slack > 0 it also stops,
// from the second digit on (a first-digit bucket is too coarse a bound),
// once the bucket holds at most krem + slack candidates: taking the whole
// bucket then keeps between kk and kk + slack candidates, all of them at
// least as good as every candidate left out. A pass after the first that
// leaves more than abort_cnt candidates in the boundary bucket ends the
// selection unresolved (stopped = false), for callers that only want a
// cheap answer.
//
// Work saving: every pass also records the AND / OR of the candidate keys
// it visits, and pass 1 their positions in `cb` when they fit; later passes
// then visit only those positions, a digit on which all candidates of the
// previous pass agree is folded without a pass, and at most kFinishMax
// boundary candidates are resolved by counting.
// Each pass takes one barrier: every warp finds the bucket itself. `pass`
// is the block's pass counter (see PassSlot). Requires at least kk
// candidates. Block-wide.
template <class Key, int KEY_BITS, int NT, class Get>
__device__ Radix<Key> radix_select(Ctrl& ctl, uint32_t& pass, uint32_t count, const uint16_t* dom, uint32_t dom_n,
                                   uint32_t kk, uint32_t slack, uint32_t abort_cnt, CandBuf& cb, Get&& get)
{
  constexpr int P = KEY_BITS / kDigitBits;
  constexpr int UNR = 4;
  Radix<Key> r{(Key)0, (Key)0, kk, 0u, false};
  const uint32_t span = dom ? dom_n : count;
  const bool can_compact = cb.pos != nullptr;
  bool compacted = false;
  uint32_t ncand = 0;
  Key diff = ~(Key)0; // digits that may differ among the remaining candidates
  Key kand_v = 0;
#ifdef SEGTOPK_STATS
  long long t_pass = clock64();
#endif
  for (int p = 0; p < P; ++p) {
    const int shift = KEY_BITS - kDigitBits * (p + 1);
    const Key dmask = (Key)(kBuckets - 1) << shift;
    if (p >= 1 && !(diff & dmask)) {
      // every remaining candidate has the same digit here: fold it without a pass
      r.prefix |= kand_v & dmask;
      r.mask |= dmask;
      continue;
    }
    PassSlot& sl = ctl.slot[pass % 3];
    uint32_t* h = sl.hist;
    const bool rec = true; // record AND / OR (every pass: a digit its candidates share is folded next)
    const bool collect = p == 1 && can_compact;
    const uint32_t n_visit = compacted ? ncand : span;
    Key ta = ~(Key)0, to = (Key)0;
    for (uint32_t base = 0; base < n_visit; base += NT * UNR) {
      Key key[UNR];
      uint32_t e[UNR];
      bool on[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const uint32_t i = base + (uint32_t)u * NT + threadIdx.x;
        on[u] = false;
        key[u] = 0;
        e[u] = 0;
        if (i < n_visit) {
          e[u] = compacted ? (uint32_t)cb.pos[i] : (dom ? (uint32_t)dom[i] : i);
          on[u] = get(e[u], key[u]) && (key[u] & r.mask) == r.prefix;
        }
      }
      uint32_t nc = 0;
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (on[u]) {
          atomicAdd(&h[(uint32_t)(key[u] >> shift) & (kBuckets - 1)], 1u);
          ta &= key[u];
          to |= key[u];
          ++nc;
        }
      }
      if (collect && nc) {
        uint32_t slot = atomicAdd(&sl.ncand, nc);
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          if (on[u]) {
            if (slot < cb.cap)
              cb.pos[slot] = (uint16_t)e[u];
            ++slot;
          }
        }
      }
    }
    if (rec)
      fold_and_or(sl.and_w, sl.or_w, ta, to);
    clear_slot<NT>(ctl.slot[(pass + 1) % 3]);
    __syncthreads();
    uint32_t b, before, cnt;
    find_bucket_warp(h, r.krem, b, before, cnt);
    if (rec) {
      kand_v = read_word<Key>(sl.and_w);
      diff = kand_v ^ read_word<Key>(sl.or_w);
    }
    if (collect) {
      ncand = sl.ncand;
      compacted = ncand <= cb.cap;
    }
    ++pass;
    r.krem -= before;
    r.cnt = cnt;
    r.prefix |= (Key)b << shift;
    r.mask |= dmask;
    if (cnt == r.krem || (p >= 1 && cnt - r.krem <= slack)) {
      r.stopped = true;
      break;
    }
    if (p >= 1 && cnt > abort_cnt)
      break;
    if (compacted && cnt <= kFinishMax && p + 1 < P) {
      // few candidates left: resolve the boundary key by counting (the slot
      // of the pass just done holds the staging counter)
      Key v;
      uint32_t less, eq;
#ifdef SEGTOPK_STATS
      SEGTOPK_STAT_ADD(kStatSelPasses, clock64() - t_pass);
      t_pass = clock64();
#endif
      finish_by_count<Key, NT>(reinterpret_cast<Key*>(ctl.fin), &ctl.slot[(pass + 2) % 3].nfin, cb.pos, ncand,
                               r.prefix, r.mask, r.krem, get, v, less, eq);
#ifdef SEGTOPK_STATS
      SEGTOPK_STAT_ADD(kStatSelFinish, clock64() - t_pass);
      t_pass = 0;
#endif
      r.prefix = v;
      r.mask = ~(Key)0;
      r.krem -= less;
      r.cnt = eq;
      r.stopped = eq - r.krem <= slack;
      break;
    }
  }
#ifdef SEGTOPK_STATS
  if (t_pass)
    SEGTOPK_STAT_ADD(kStatSelPasses, clock64() - t_pass);
#endif
  cb.n = compacted ? ncand : ~0u;
  return r;
}

// Preference index: smaller is preferred among equal keys.
__device__ __forceinline__ uint32_t pref_index(uint32_t idx, bool prefer_larger)
{
  return prefer_larger ? ~idx : idx;
}

// Which list entries form the k best: (rank & mask) < prefix are strictly
// better than the boundary ("front"); among the boundary candidates
// ((rank & mask) == prefix) those with (pref_index & imask) <= iprefix are
// taken. imask == 0 takes every boundary candidate -- or, with take > 0,
// the first `take` of them in order of arrival (a compaction counts them):
// the tie choice of the not_guaranteed determinism mode, where any subset of
// the ties is valid ("Top-K: Determinism, Tie-Breaking, and Output
// Ordering", "Determinism" table).
template <class Rank>
struct Selection {
  Rank prefix, mask;
  uint32_t iprefix, imask;
  uint32_t n;    // entries selected
  uint32_t take; // > 0: boundary entries taken by arrival, at most this many
  // 0: not selected, 1: front, 2: selected boundary entry
  __device__ __forceinline__ int classify(Rank r, uint32_t pidx) const
  {
    const Rank mr = r & mask;
    if (mr < prefix)
      return 1;
    return (mr == prefix && (pidx & imask) <= iprefix) ? 2 : 0;
  }
};

// Boundary ties by source index: among entries with (rank & mask) == prefix,
// choose the q preferred ones (0 < q < their count) by a second radix
// selection on the preference index, which is unique within a segment. If
// the rank selection left the boundary candidates in `cb`, only those are
// visited.
template <class TR, int NT>
__device__ void select_ties(Ctrl& ctl, uint32_t& pass, const Src<typename TR::Raw>& src, uint32_t q,
                            typename TR::Rank dirmask, bool prefer_larger, Selection<typename TR::Rank>& s,
                            CandBuf& cb)
{
  using Rank = typename TR::Rank;
  const Rank prefix = s.prefix, mask = s.mask;
  const bool use = cb.pos != nullptr && cb.n != ~0u;
  CandBuf none{nullptr, 0u, ~0u};
  const Radix<uint32_t> ri = radix_select<uint32_t, 32, NT>(
    ctl, pass, src.size(), use ? cb.pos : nullptr, use ? cb.n : 0u, q, 0u, ~0u, use ? none : cb, [&](uint32_t e, uint32_t& key) {
      key = pref_index(src.index(e), prefer_larger);
      return (TR::rank(src.key(e), dirmask) & mask) == prefix;
    });
  s.iprefix = ri.prefix;
  s.imask = ri.mask;
}

// Boundary ties when every entry of `src` is a ring key (no list entries):
// position order is source-index order, so the q preferred ties are the
// first q (prefer_smaller) or last q (prefer_larger) ties by position. Each
// thread counts the ties in its run of consecutive entries, a block scan
// over the counts gives every run's first tie number, and the thread
// holding the q-th preferred tie publishes its preference index, which
// becomes the tie threshold ("Implement Segmented TopK using
// Thread-Block-Clusters", section 5: ties taken in index order by prefix
// scans). Block-wide.
template <class TR, int NT>
__device__ __forceinline__ void select_ties_ordered(Ctrl& ctl, const Src<typename TR::Raw>& src, uint32_t q,
                                                 typename TR::Rank dirmask, bool prefer_larger,
                                                 Selection<typename TR::Rank>& s)
{
  using Rank = typename TR::Rank;
  const Rank prefix = s.prefix, mask = s.mask;
  const uint32_t n = src.ext_count;
  const uint32_t per = (n + NT - 1) / NT;
  const uint32_t e0 = min(n, threadIdx.x * per), e1 = min(n, e0 + per);
  uint32_t c = 0;
  for (uint32_t e = e0; e < e1; ++e)
    c += (TR::rank(src.ext_raw[e], dirmask) & mask) == prefix ? 1u : 0u;
  // block exclusive scan of c over threads in position order
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t incl = warp_inclusive_sum(c);
  if (lane == 31)
    ctl.red[warp] = incl;
  __syncthreads();
  uint32_t before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const uint32_t t = (uint32_t)ctl.red[w];
    before += (uint32_t)w < warp ? t : 0u;
    total += t;
  }
  const uint32_t excl = before + incl - c;
  // 0-based position (ascending) of the q-th preferred tie
  const uint32_t target = prefer_larger ? total - q : q - 1;
  if (target >= excl && target < excl + c) {
    uint32_t r = excl;
    for (uint32_t e = e0; e < e1; ++e) {
      if ((TR::rank(src.ext_raw[e], dirmask) & mask) == prefix) {
        if (r == target)
          ctl.res[0] = pref_index(src.ext_idx0 + e, prefer_larger);
        ++r;
      }
    }
  }
  __syncthreads();
  s.iprefix = ctl.res[0];
  s.imask = ~0u;
  __syncthreads(); // ctl.red and ctl.res are free again
}

// The kk best of the entries of `src` (size > kk > 0) in one CTA -- or,
// with slack > 0, between kk and kk + slack entries that include them: a
// radix selection on the rank code, then, if more boundary entries tie than
// are needed, one on the preference index.
template <class TR, int NT>
__device__ Selection<typename TR::Rank> block_select(Ctrl& ctl, uint32_t& pass, const Src<typename TR::Raw>& src,
                                                     uint32_t kk, uint32_t slack, typename TR::Rank dirmask,
                                                     bool prefer_larger, CandBuf cb, bool tie_any)
{
  using Rank = typename TR::Rank;
  const Radix<Rank> rr = radix_select<Rank, TR::kRankBits, NT>(ctl, pass, src.size(), nullptr, 0u, kk, slack, ~0u, cb,
                                                               [&](uint32_t e, Rank& key) {
                                                                 key = TR::rank(src.key(e), dirmask);
                                                                 return true;
                                                               });
  Selection<Rank> s{rr.prefix, rr.mask, 0u, 0u, kk};
  if (rr.stopped) // the whole boundary bucket is taken
    s.n = kk - rr.krem + rr.cnt;
  else if (src.count == 0) // every rank digit resolved, more than krem ties, ring keys only
    select_ties_ordered<TR, NT>(ctl, src, rr.krem, dirmask, prefer_larger, s);
  else if (tie_any) // more than krem ties and any of them will do: the first to arrive
    s.take = rr.krem;
  else // every rank digit resolved and more than krem entries share the boundary rank
    select_ties<TR, NT>(ctl, pass, src, rr.krem, dirmask, prefer_larger, s, cb);
  return s;
}

// Walks list entries [0, count); classify(e, raw, idx, rank) returns 0 (skip),
// 1 or 2. For every entry of class 1 or 2 it calls
//   sink(e, raw, idx, rank, cls, rank1, rank2)
// where rank1 / rank2 count the class-1 / class-2 entries before e (warp
// ballots over a warp's contiguous run of 128 entries, a block scan across
// warps). Returns the class totals. The sink runs after a barrier that
// follows every thread's reads of the current tile, so it may overwrite list
// slots at or before the tile.
template <class TR, int NT, class Classify, class Sink>
__device__ uint2 scan_list(Ctrl& ctl, const Src<typename TR::Raw>& src, typename TR::Rank dirmask,
                           Classify&& classify, Sink&& sink)
{
  const uint32_t count = src.size();
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  constexpr int NW = NT / 32;
  constexpr int R = 4; // rounds of 32 entries per warp and tile
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  uint32_t seen1 = 0, seen2 = 0;
  int buf = 0;
  for (uint32_t tile = 0; tile < count; tile += NT * R) {
    Raw kr[R];
    uint32_t ki[R];
    Rank rk[R];
    uint32_t b1[R], b2[R];
    uint32_t w1 = 0, w2 = 0;
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const uint32_t e = tile + warp * (32 * R) + q * 32 + lane;
      const bool valid = e < count;
      kr[q] = valid ? src.key(e) : Raw(0);
      ki[q] = valid ? src.index(e) : 0u;
      rk[q] = TR::rank(kr[q], dirmask);
      const int c = valid ? classify(e, kr[q], ki[q], rk[q]) : 0;
      b1[q] = __ballot_sync(kFull, c == 1);
      b2[q] = __ballot_sync(kFull, c == 2);
      w1 += __popc(b1[q]);
      w2 += __popc(b2[q]);
    }
    if (lane == 0)
      ctl.scan_tot[buf][warp] = (uint64_t)w1 | ((uint64_t)w2 << 32);
    __syncthreads();
    uint32_t f1 = seen1, f2 = seen2, t1 = 0, t2 = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint64_t v = ctl.scan_tot[buf][w];
      if (w < (int)warp) {
        f1 += (uint32_t)v;
        f2 += (uint32_t)(v >> 32);
      }
      t1 += (uint32_t)v;
      t2 += (uint32_t)(v >> 32);
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const bool is1 = (b1[q] >> lane) & 1u;
      const bool is2 = (b2[q] >> lane) & 1u;
      if (is1 || is2)
        sink(tile + warp * (32 * R) + q * 32 + lane, kr[q], ki[q], rk[q], is1 ? 1 : 2,
             f1 + __popc(b1[q] & lt), f2 + __popc(b2[q] & lt));
      f1 += __popc(b1[q]);
      f2 += __popc(b2[q]);
    }
    seen1 += t1;
    seen2 += t2;
    buf ^= 1;
  }
  __syncthreads(); // sink writes visible; scan_tot free for the next walk
  return make_uint2(seen1, seen2);
}

// Block-wide maximum of a rank value (every thread gets the result).
template <class Rank, int NT>
__device__ __forceinline__ Rank block_max(Ctrl& ctl, Rank v)
{
  v = warp_max(v);
  if (lane_id() == 0)
    ctl.red[threadIdx.x >> 5] = (uint64_t)v;
  __syncthreads();
  Rank m = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const Rank x = (Rank)ctl.red[w];
    m = x > m ? x : m;
  }
  __syncthreads(); // ctl.red is free again
  return m;
}

// The worst (largest (rank, preference index)) of `count` list entries.
// Block-wide; every thread gets the result.
template <class TR, int NT>
__device__ __forceinline__ void list_worst(Ctrl& ctl, const typename TR::Raw* raw, const uint32_t* idx,
                                           uint32_t count, typename TR::Rank dirmask, bool prefer_larger,
                                           uint64_t& w_rank, uint64_t& w_pidx)
{
  using Rank = typename TR::Rank;
  if constexpr (TR::kRankBits <= 32) {
    uint64_t mx = 0;
    for (uint32_t e = threadIdx.x; e < count; e += NT) {
      const uint64_t c = ((uint64_t)TR::rank(raw[e], dirmask) << 32) | pref_index(idx[e], prefer_larger);
      mx = c > mx ? c : mx;
    }
    mx = block_max<uint64_t, NT>(ctl, mx);
    w_rank = mx >> 32;
    w_pidx = mx & 0xffffffffull;
  } else {
    Rank mr = 0;
    for (uint32_t e = threadIdx.x; e < count; e += NT) {
      const Rank r = TR::rank(raw[e], dirmask);
      mr = r > mr ? r : mr;
    }
    mr = block_max<Rank, NT>(ctl, mr);
    uint32_t mp = 0;
    for (uint32_t e = threadIdx.x; e < count; e += NT) {
      const uint32_t pi = pref_index(idx[e], prefer_larger);
      if (TR::rank(raw[e], dirmask) == mr)
        mp = pi > mp ? pi : mp;
    }
    mp = block_max<uint32_t, NT>(ctl, mp);
    w_rank = (uint64_t)mr;
    w_pidx = mp;
  }
}

// Entries kept by a compaction: their number and their largest rank, and
// the block's pass counter after the selection.
template <class Rank>
struct Kept {
  Rank max_rank;
  uint32_t n;
  uint32_t pass;
};

// Writes the entries of `src` that `s` selects to dst[0, cap) in no
// particular order (warp-aggregated atomic positions, one pass, no scan),
// and returns their number and largest rank. `pass` is the pass counter
// after the selection: the slot of its last pass holds the counters. dst
// must not overlap src's arrays. Block-wide; ends with a barrier.
template <class TR, int NT>
__device__ __forceinline__ Kept<typename TR::Rank> select_into(Ctrl& ctl, uint32_t pass,
                                                               const Src<typename TR::Raw>& src,
                                                               const Selection<typename TR::Rank>& s,
                                                               typename TR::Raw* dst_raw, uint32_t* dst_idx,
                                                               uint32_t cap, typename TR::Rank dirmask,
                                                               bool prefer_larger)
{
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  PassSlot& sl = ctl.slot[(pass + 2) % 3];
  Rank mx = 0;
  const uint32_t n = src.size();
#ifdef SEGTOPK_STATS
  const long long t_compact = clock64();
#endif
  for (uint32_t base = 0; base < n; base += NT) {
    const uint32_t e = base + threadIdx.x;
    bool keep = false;
    Raw kr = 0;
    uint32_t ki = 0;
    Rank rk = 0;
    int cls = 0;
    if (e < n) {
      kr = src.key(e);
      ki = src.index(e);
      rk = TR::rank(kr, dirmask);
      cls = s.classify(rk, pref_index(ki, prefer_larger));
      keep = cls != 0;
    }
    if (s.take) {
      // boundary entries by arrival: one counter add per warp and round
      const uint32_t tb = __ballot_sync(kFull, cls == 2);
      if (tb) {
        uint32_t tbase = 0;
        if (lane_id() == 0)
          tbase = atomicAdd(&sl.ties, __popc(tb));
        tbase = __shfl_sync(kFull, tbase, 0);
        if (cls == 2)
          keep = tbase + __popc(tb & lanemask_lt()) < s.take;
      }
    }
    const uint32_t bal = __ballot_sync(kFull, keep);
    if (bal) {
      uint32_t wb = 0;
      if (lane_id() == 0)
        wb = atomicAdd(&sl.kept, __popc(bal));
      const uint32_t pos = __shfl_sync(kFull, wb, 0) + __popc(bal & lanemask_lt());
      if (keep && pos < cap) { // pos < cap always holds for a valid selection; guards dst
        dst_raw[pos] = kr;
        dst_idx[pos] = ki;
        mx = rk > mx ? rk : mx;
      }
    }
  }
  mx = warp_max(mx);
  if (lane_id() == 0 && mx != 0)
    atomicMax(&sl.kmax, (unsigned long long)mx);
  __syncthreads(); // publishes dst and the counters
  SEGTOPK_STAT_ADD(kStatSelCompact, clock64() - t_compact);
  return Kept<Rank>{(Rank)sl.kmax, s.n < cap ? s.n : cap, pass};
}

// Keep the kk best entries of `src` (size > kk > 0) -- with slack > 0,
// between kk and kk + slack entries that include them -- in dst, which holds
// kk + slack entries. Returns the number kept and their largest rank: later
// keys (which come after every kept one in preference order) are accepted
// only below it.
template <class TR, int NT>
__device__ __forceinline__ Kept<typename TR::Rank> trim_into(Ctrl& ctl, uint32_t pass, const Src<typename TR::Raw> src,
                                                          typename TR::Raw* dst_raw, uint32_t* dst_idx, uint32_t kk,
                                                          uint32_t slack, typename TR::Rank dirmask,
                                                          bool prefer_larger, CandBuf cb, bool tie_any)
{
  const Selection<typename TR::Rank> s =
    block_select<TR, NT>(ctl, pass, src, kk, slack, dirmask, prefer_larger, cb, tie_any);
  return select_into<TR, NT>(ctl, pass, src, s, dst_raw, dst_idx, kk + slack, dirmask, prefer_larger);
}

// The kk best of ring keys only (src.count == 0) when their kk-th key is
// expected to lie in a block of keys tied at rank e (a speculative
// selection just met that block): one count of the keys better than e and
// equal to it, and if the kk-th key is indeed a tie, the better keys and the
// first kk - better ties in preference order (select_ties_ordered) written
// to dst -- no digit passes. Returns n == 0 if the kk-th key is not a tie.
template <class TR, int NT>
__device__ __forceinline__ Kept<typename TR::Rank> tie_block_into(Ctrl& ctl, uint32_t pass,
                                                                  const Src<typename TR::Raw>& src,
                                                                  typename TR::Rank e, uint32_t kk,
                                                                  typename TR::Raw* dst_raw, uint32_t* dst_idx,
                                                                  uint32_t cap, typename TR::Rank dirmask,
                                                                  bool prefer_larger)
{
  using Rank = typename TR::Rank;
  if (threadIdx.x == 0) {
    // select_into counts in the slot of the last digit pass; none ran here
    PassSlot& sl = ctl.slot[(pass + 2) % 3];
    sl.kept = 0;
    sl.ties = 0;
    sl.kmax = 0;
  }
  const uint32_t n = src.ext_count;
  uint32_t f = 0, t = 0;
  for (uint32_t i = threadIdx.x; i < n; i += NT) {
    const Rank r = TR::rank(src.ext_raw[i], dirmask);
    f += r < e ? 1u : 0u;
    t += r == e ? 1u : 0u;
  }
  f = __reduce_add_sync(kFull, f);
  t = __reduce_add_sync(kFull, t);
  if (lane_id() == 0)
    ctl.red[threadIdx.x >> 5] = ((uint64_t)f << 32) | t;
  __syncthreads();
  uint32_t front = 0, ties = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    front += (uint32_t)(ctl.red[w] >> 32);
    ties += (uint32_t)ctl.red[w];
  }
  __syncthreads(); // ctl.red is free again
  if (!(front < kk && kk <= front + ties && kk <= cap))
    return Kept<Rank>{(Rank)0, 0u, pass};
  Selection<Rank> s{e, ~(Rank)0, 0u, 0u, kk};
  select_ties_ordered<TR, NT>(ctl, src, kk - front, dirmask, prefer_larger, s);
  return select_into<TR, NT>(ctl, pass, src, s, dst_raw, dst_idx, cap, dirmask, prefer_larger);
}

// A speculative first bound from a sample of a slice: the smallest rank
// edge with at least mm sample entries at or below it (mm is below the
// number the slice needs), found by a digit selection that may stop early
// with up to 2 mm entries. Every sample entry with rank <= edge is written
// to dst (capacity cap); the caller then accepts later keys with rank <=
// edge only, and must verify at the end that the slice produced enough
// entries. Fails (ok = false, nothing written) when the entries at the
// boundary rank are too many (heavy ties: given up as soon as a digit pass
// after the first leaves more than 8 mm + 64 of them) or edge is the worst
// rank.
template <class Rank>
struct Spec {
  bool ok;
  Rank edge;
  uint32_t n;
  uint32_t pass;
  bool tie_block; // failed on a block of keys tied at rank `edge` (an exact rank)
};
template <class TR, int NT>
__device__ __forceinline__ Spec<typename TR::Rank> spec_into(Ctrl& ctl, uint32_t pass, const Src<typename TR::Raw> src,
                                                          typename TR::Raw* dst_raw, uint32_t* dst_idx, uint32_t mm,
                                                          uint32_t cap, typename TR::Rank dirmask, CandBuf cb)
{
  using Rank = typename TR::Rank;
  constexpr Rank kWorst = (TR::kRankBits == 64) ? ~(Rank)0 : (Rank)(((uint64_t)1 << TR::kRankBits) - 1);
  Selection<Rank> s;
  Rank edge;
  uint32_t total;
  bool ok;
  if constexpr (TR::kRankBits == 64) {
    // 64-bit ranks: the high word is resolution enough for a first bound
    const Radix<uint32_t> rr = radix_select<uint32_t, 32, NT>(ctl, pass, src.size(), nullptr, 0u, mm, mm,
                                                              8u * mm + 64u, cb, [&](uint32_t e, uint32_t& key) {
                                                                key = (uint32_t)(TR::rank(src.key(e), dirmask) >> 32);
                                                                return true;
                                                              });
    const uint32_t edge_hi = rr.prefix | ~rr.mask;
    edge = ((Rank)edge_hi << 32) | 0xffffffffull;
    total = mm - rr.krem + rr.cnt;
    ok = rr.stopped;
    s = Selection<Rank>{(Rank)rr.prefix << 32, (Rank)rr.mask << 32, 0u, 0u, total};
  } else {
    const Radix<Rank> rr = radix_select<Rank, TR::kRankBits, NT>(ctl, pass, src.size(), nullptr, 0u, mm, mm,
                                                                 8u * mm + 64u, cb, [&](uint32_t e, Rank& key) {
                                                                   key = TR::rank(src.key(e), dirmask);
                                                                   return true;
                                                                 });
    edge = rr.prefix | (~rr.mask & kWorst);
    total = mm - rr.krem + rr.cnt;
    ok = rr.stopped;
    s = Selection<Rank>{rr.prefix, rr.mask, 0u, 0u, total}; // the whole boundary bucket
  }
  if (!ok || edge == kWorst || total > cap)
    return Spec<Rank>{false, (Rank)0, 0u, pass, false};
  const Kept<Rank> kp = select_into<TR, NT>(ctl, pass, src, s, dst_raw, dst_idx, cap, dirmask, false);
  return Spec<Rank>{true, edge, kp.n, pass, false};
}

// The speculative first bound for a small target (mm <= 32) and a sample of
// ring keys only (at most KPT per thread), without digit passes: every
// thread sorts its sample keys in registers, every warp extracts its
// min(mm, kSpecDepth) smallest by repeated warp minimums, and warp 0 takes
// the mm-th smallest of the warps' lists, two per lane, the same way. That
// is the sample's mm-th smallest unless one warp holds more than kSpecDepth
// of the sample's mm smallest; the edge is then a little worse, and still
// at least mm sample keys lie at or below it. Selection keys are 32 bits:
// the rank, or its high word for 64-bit ranks (resolution enough for a first
// bound). Every sample key at or below the edge is written to dst, as
// spec_into does; `stage` is 1 KiB of free shared memory. Fails (nothing
// usable written) on heavy ties at the edge (the target's value also at half
// the target, or more than 2 mm + 64 keys kept) or an edge at the worst rank.
constexpr uint32_t kSpecDepth = 8;
template <class TR, int NT, int KPT>
__device__ __forceinline__ Spec<typename TR::Rank> spec_small(Ctrl& ctl, uint32_t pass, const typename TR::Raw* sample,
                                                              uint32_t idx0, uint32_t ns, uint32_t mm,
                                                              typename TR::Raw* dst_raw, uint32_t* dst_idx,
                                                              uint32_t cap, typename TR::Rank dirmask,
                                                              uint32_t* stage)
{
  using Rank = typename TR::Rank;
  constexpr int NW = NT / 32;
  static_assert(NW * kSpecDepth <= 64, "the warps' lists fit two per lane");
  static_assert(KPT == 4 || KPT == 8, "sample keys per thread");
  auto key32 = [&](uint32_t e) -> uint32_t {
    const Rank r = TR::rank(sample[e], dirmask);
    if constexpr (TR::kRankBits == 64)
      return (uint32_t)(r >> 32);
    else
      return (uint32_t)r;
  };
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
#ifdef SEGTOPK_STATS
  long long t_phase = clock64();
  auto phase_done = [&](int stat) {
    SEGTOPK_STAT_ADD(stat, clock64() - t_phase);
    t_phase = clock64();
  };
#else
  auto phase_done = [](int) {};
#endif
  uint32_t v[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const uint32_t e = (uint32_t)i * NT + threadIdx.x;
    v[i] = e < ns ? key32(e) : ~0u;
  }
  // odd-even transposition sort of the thread's keys
#pragma unroll
  for (int round = 0; round < KPT; ++round) {
#pragma unroll
    for (int i = round & 1; i + 1 < KPT; i += 2) {
      const uint32_t lo = min(v[i], v[i + 1]), hi = max(v[i], v[i + 1]);
      v[i] = lo;
      v[i + 1] = hi;
    }
  }
  // the warp's rw smallest, in order (the rest of its list: the worst key)
  const uint32_t rw = mm < kSpecDepth ? mm : kSpecDepth;
  for (uint32_t it = 0; it < kSpecDepth; ++it) {
    uint32_t mn = ~0u;
    if (it < rw) {
      mn = __reduce_min_sync(kFull, v[0]);
      const uint32_t win = __ffs(__ballot_sync(kFull, v[0] == mn)) - 1;
      if (lane == win) {
#pragma unroll
        for (int i = 0; i + 1 < KPT; ++i)
          v[i] = v[i + 1];
        v[KPT - 1] = ~0u;
      }
    }
    if (lane == 0)
      stage[warp * kSpecDepth + it] = mn;
  }
  if (threadIdx.x == 0)
    ctl.spec_kept = 0;
  __syncthreads();
  phase_done(kStatSpecWarp);
  // warp 0: the mm-th smallest of the warps' lists (two keys per lane, slots
  // lane and lane + 32): a larger target by counting -- a key's place in the
  // order (key, slot) is the number of keys before it, 64 independent
  // comparisons -- a small one by repeated warp minimums
  if (warp == 0) {
    const uint32_t x0 = lane < (uint32_t)(NW * kSpecDepth) ? stage[lane] : ~0u;
    const uint32_t x1 = lane + 32u < (uint32_t)(NW * kSpecDepth) ? stage[lane + 32u] : ~0u;
    uint32_t lo = min(x0, x1), hi = max(x0, x1);
    uint32_t edge = ~0u, mid = ~0u;
    if (mm >= 16u) {
      uint32_t r0 = 0, r1 = 0;
#pragma unroll 8
      for (uint32_t j = 0; j < 32; ++j) {
        const uint32_t y0 = __shfl_sync(kFull, x0, j), y1 = __shfl_sync(kFull, x1, j);
        r0 += (uint32_t)(y0 < x0 || (y0 == x0 && j < lane)) + (uint32_t)(y1 < x0);
        r1 += (uint32_t)(y0 <= x1) + (uint32_t)(y1 < x1 || (y1 == x1 && j < lane));
      }
      auto at_place = [&](uint32_t q) {
        const uint32_t b0 = __ballot_sync(kFull, r0 == q), b1 = __ballot_sync(kFull, r1 == q);
        return b0 ? __shfl_sync(kFull, x0, __ffs(b0) - 1) : __shfl_sync(kFull, x1, __ffs(b1) - 1);
      };
      edge = at_place(mm - 1);
      mid = at_place((mm - 1) / 2);
    }
    for (uint32_t it = 0; mm < 16u && it < mm; ++it) {
      const uint32_t mn = __reduce_min_sync(kFull, lo);
      const uint32_t win = __ffs(__ballot_sync(kFull, lo == mn)) - 1;
      edge = mn;
      if (it == (mm - 1) / 2)
        mid = mn;
      if (lane == win) {
        lo = hi;
        hi = ~0u;
      }
    }
    if (lane == 0) {
      ctl.res[0] = edge;
      ctl.res[1] = (mm > 2u && mid == edge) ? 1u : 0u; // the target's value fills half of it: a tie block
    }
  }
  __syncthreads();
  phase_done(kStatSpecMerge);
  const uint32_t e32 = ctl.res[0];
  if (ctl.res[1]) {
    __syncthreads(); // ctl.res and the stage are free again
    return Spec<Rank>{false, (Rank)e32, 0u, pass, TR::kRankBits <= 32};
  }
  // every sample key at or below the edge into dst (warp-aggregated slots)
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const uint32_t e = (uint32_t)i * NT + threadIdx.x;
    const bool keep = e < ns && key32(e) <= e32;
    const uint32_t bal = __ballot_sync(kFull, keep);
    if (bal) {
      uint32_t wb = 0;
      if (lane == 0)
        wb = atomicAdd(&ctl.spec_kept, __popc(bal));
      const uint32_t pos = __shfl_sync(kFull, wb, 0) + __popc(bal & lanemask_lt());
      if (keep && pos < cap) {
        dst_raw[pos] = sample[e];
        dst_idx[pos] = idx0 + e;
      }
    }
  }
  __syncthreads();
  const uint32_t kept = ctl.spec_kept;
  __syncthreads(); // ctl.res and the stage are free again
  phase_done(kStatSpecKeep);
  Rank edge;
  if constexpr (TR::kRankBits == 64)
    edge = ((Rank)e32 << 32) | 0xffffffffull;
  else
    edge = (Rank)e32;
  constexpr Rank kWorst = (TR::kRankBits == 64) ? ~(Rank)0 : (Rank)(((uint64_t)1 << TR::kRankBits) - 1);
  const bool ties = kept > 2u * mm + 64u || kept > cap;
  const bool ok = edge < kWorst && !ties;
  return Spec<Rank>{ok, edge, kept, pass, ties && TR::kRankBits <= 32};
}

// ---------------------------------------------------------------------------
// Sorting the selected items (up to 2048) for sorted output: a bitonic
// network over registers, warp shuffles and, for the widest strides,
// shared memory.
// ---------------------------------------------------------------------------
// Shared-memory bitonic sort of n2 (a power of two) keys with payloads.
// Compare-exchange pairs: thread i of a stage takes lo = i + (i & ~(stride-1))
// and hi = lo + stride. A warp's 32 consecutive i cover one aligned block of
// 64 elements, so stages with stride <= 32 only exchange inside blocks the
// warp owns and need only a warp barrier; wider strides take block barriers
// (10 of the 55 stages of a 1024-element sort).
template <int NT>
__device__ void bitonic_sort_u64(uint64_t* key, uint32_t* pay, uint32_t n2)
{
  bool warp_phase = false; // the last stage synchronised its warp only
  for (uint32_t size = 2; size <= n2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      const bool block_stage = stride > 32;
      if (block_stage && warp_phase)
        __syncthreads();
      for (uint32_t i = threadIdx.x; i < (n2 >> 1); i += NT) {
        const uint32_t lo = i + (i & ~(stride - 1));
        const uint32_t hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = key[lo], b = key[hi];
        if ((a > b) == up) {
          key[lo] = b;
          key[hi] = a;
          const uint32_t t = pay[lo];
          pay[lo] = pay[hi];
          pay[hi] = t;
        }
      }
      if (block_stage)
        __syncthreads();
      else
        __syncwarp();
      warp_phase = !block_stage;
    }
  }
  if (warp_phase)
    __syncthreads();
}

template <int NT>
__device__ void bitonic_sort_u128(uint64_t* khi, uint64_t* klo, uint32_t n2)
{
  bool warp_phase = false;
  for (uint32_t size = 2; size <= n2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      const bool block_stage = stride > 32;
      if (block_stage && warp_phase)
        __syncthreads();
      for (uint32_t i = threadIdx.x; i < (n2 >> 1); i += NT) {
        const uint32_t lo = i + (i & ~(stride - 1));
        const uint32_t hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t ah = khi[lo], al = klo[lo], bh = khi[hi], bl = klo[hi];
        const bool gt = ah > bh || (ah == bh && al > bl);
        if (gt == up) {
          khi[lo] = bh;
          klo[lo] = bl;
          khi[hi] = ah;
          klo[hi] = al;
        }
      }
      if (block_stage)
        __syncthreads();
      else
        __syncwarp();
      warp_phase = !block_stage;
    }
  }
  if (warp_phase)
    __syncthreads();
}

// Threads a block sort spreads its elements over (the CTA size).
constexpr uint32_t kSortLanes = 256;

// In-thread compare-exchange stage of the register sort (stride S < EPT).
template <int EPT, int S>
__device__ __forceinline__ void sort_in_thread(uint64_t (&a)[EPT], uint64_t (&b)[EPT], uint32_t size)
{
#pragma unroll
  for (int r = 0; r < EPT; ++r) {
    if ((r & S) == 0) {
      const int r2 = r | S;
      const uint32_t e = threadIdx.x * (uint32_t)EPT + (uint32_t)r;
      const bool up = (e & size) == 0;
      const bool gt = a[r] > a[r2] || (a[r] == a[r2] && b[r] > b[r2]);
      if (gt == up) {
        const uint64_t ta = a[r], tb = b[r];
        a[r] = a[r2];
        b[r] = b[r2];
        a[r2] = ta;
        b[r2] = tb;
      }
    }
  }
}

// Bitonic sort of EPT * NT elements (a, b), ascending by a then b. Thread t
// holds elements t*EPT .. t*EPT+EPT-1 in registers: strides below EPT are
// exchanged inside the thread, strides below 32*EPT between lanes of a warp
// by shuffles, and wider ones through shared memory (s1, s2: one word each
// per element) with block barriers -- 6 of the 55 stages for 1024 elements.
template <int NT, int EPT>
__device__ __forceinline__ void reg_bitonic_sort(uint64_t (&a)[EPT], uint64_t (&b)[EPT], uint64_t* s1, uint64_t* s2)
{
  constexpr uint32_t N = (uint32_t)(EPT * NT);
  const uint32_t t = threadIdx.x;
  // fully unrolled: every stride is a constant, so each stage compiles to
  // straight register, shuffle or shared-memory code
#pragma unroll
  for (uint32_t size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < (uint32_t)EPT) {
        if (stride == 4)
          sort_in_thread<EPT, (EPT > 4 ? 4 : 0)>(a, b, size);
        else if (stride == 2)
          sort_in_thread<EPT, (EPT > 2 ? 2 : 0)>(a, b, size);
        else
          sort_in_thread<EPT, (EPT > 1 ? 1 : 0)>(a, b, size);
        continue;
      }
      const bool lower_lane = stride < 32u * EPT ? (t & (stride / EPT)) == 0 : false;
      if (stride >= 32u * EPT) {
#pragma unroll
        for (int r = 0; r < EPT; ++r) {
          s1[t * EPT + r] = a[r];
          s2[t * EPT + r] = b[r];
        }
        __syncthreads();
      }
#pragma unroll
      for (int r = 0; r < EPT; ++r) {
        const uint32_t e = t * (uint32_t)EPT + (uint32_t)r;
        uint64_t oa, ob;
        bool lower;
        if (stride < 32u * EPT) {
          oa = __shfl_xor_sync(kFull, a[r], stride / EPT);
          ob = __shfl_xor_sync(kFull, b[r], stride / EPT);
          lower = lower_lane;
        } else {
          oa = s1[e ^ stride];
          ob = s2[e ^ stride];
          lower = (e & stride) == 0;
        }
        const bool up = (e & size) == 0;
        const bool other_less = oa < a[r] || (oa == a[r] && ob < b[r]);
        if ((lower == up) == other_less) {
          a[r] = oa;
          b[r] = ob;
        }
      }
      if (stride >= 32u * EPT)
        __syncthreads(); // s1 / s2 are rewritten by the next such stage
    }
  }
}

__host__ __device__ inline uint32_t next_pow2(uint32_t x)
{
  uint32_t p = 1;
  while (p < x)
    p <<= 1;
  return p;
}

// Bytes of sort scratch for m items of a key whose rank has `rank_bits` bits.
__host__ __device__ inline uint32_t sort_scratch_bytes(uint32_t m, int rank_bits)
{
  const uint32_t n2 = next_pow2(m < 2 ? 2 : m);
  (void)rank_bits;
  return (n2 > kSortLanes ? n2 : kSortLanes) * 16u; // two 64-bit words per element, at least one per thread
}

// ---------------------------------------------------------------------------
// Selection and ordering by counting, for small sets (n <= kCountMax): every
// entry's position is the number of entries with a smaller key, keys being
// unique composites. Costs n^2 / NT compares per thread and two barriers,
// far below the fixed cost of digit passes on a few hundred entries.
// ---------------------------------------------------------------------------
constexpr uint32_t kCountMax = 128;
// A lone CTA's final selection takes the counting route up to this many list
// entries (one per thread: n compares per thread, two barriers), where digit
// passes and a second selection among boundary ties by source index would
// each cost a barrier and a histogram.
constexpr uint32_t kCountFinalMax = 256;

// pos[i] = #{ j < n : key_j < key_i } for unique keys (hi[i], lo[i]) (lo may
// be null for 64-bit keys). Every thread handles up to EC entries.
template <int NT, int EC>
__device__ __forceinline__ void count_ranks(const uint64_t* hi, const uint64_t* lo, uint32_t n, uint32_t* pos)
{
  uint64_t mh[EC], ml[EC];
  uint32_t c[EC];
#pragma unroll
  for (int q = 0; q < EC; ++q) {
    const uint32_t i = threadIdx.x + (uint32_t)q * NT;
    mh[q] = i < n ? hi[i] : ~0ull;
    ml[q] = (lo && i < n) ? lo[i] : ~0ull;
    c[q] = 0;
  }
  if (lo) {
    for (uint32_t j = 0; j < n; ++j) {
      const uint64_t h = hi[j], l = lo[j];
#pragma unroll
      for (int q = 0; q < EC; ++q)
        c[q] += (h < mh[q] || (h == mh[q] && l < ml[q])) ? 1u : 0u;
    }
  } else {
    for (uint32_t j = 0; j < n; ++j) {
      const uint64_t h = hi[j];
#pragma unroll
      for (int q = 0; q < EC; ++q)
        c[q] += h < mh[q] ? 1u : 0u;
    }
  }
#pragma unroll
  for (int q = 0; q < EC; ++q) {
    const uint32_t i = threadIdx.x + (uint32_t)q * NT;
    if (i < n)
      pos[i] = c[q];
  }
}

// Bytes of scratch finalize_small needs for n entries.
__host__ __device__ inline uint32_t finalize_scratch_bytes(uint32_t n) { return n * (8u + 8u + 4u); }

// The k best of n <= MAXN list entries, written to one segment's output
// slots: unsorted in selection-rank order, or stable sorted by (key, source
// index). `scratch` holds finalize_scratch_bytes(n) bytes (shared memory);
// the entries must be visible to the whole block.
template <class TR, int NT, uint32_t MAXN = kCountMax>
__device__ __forceinline__ void finalize_small(const typename TR::Raw* raw, const uint32_t* idx, uint32_t n, uint32_t k,
                                            typename TR::Rank dirmask, bool prefer_larger, bool sorted,
                                            unsigned char* scratch, typename TR::Raw* out_keys, const ValueSink& vals)
{
  constexpr int EC = (int)((MAXN + NT - 1) / NT);
  constexpr bool wide = TR::kRankBits > 32;
  uint64_t* kh = reinterpret_cast<uint64_t*>(scratch);
  uint64_t* kl = kh + n;
  uint32_t* pos = reinterpret_cast<uint32_t*>(kl + n);
  const uint32_t m = k < n ? k : n;
  // selection order: (rank, preference index)
  for (uint32_t i = threadIdx.x; i < n; i += NT) {
    const uint64_t r = (uint64_t)TR::rank(raw[i], dirmask);
    const uint32_t pi = pref_index(idx[i], prefer_larger);
    kh[i] = wide ? r : ((r << 32) | pi);
    kl[i] = pi;
  }
  __syncthreads();
  if (m < n) {
    count_ranks<NT, EC>(kh, wide ? kl : nullptr, n, pos);
    __syncthreads();
  } else {
    for (uint32_t i = threadIdx.x; i < n; i += NT)
      pos[i] = i; // every entry is selected
    __syncthreads();
  }
  if (!sorted) {
    for (uint32_t i = threadIdx.x; i < n; i += NT) {
      const uint32_t p = pos[i];
      if (p < m) {
        out_keys[p] = raw[i];
        if (vals)
          vals.put(p, idx[i]);
      }
    }
    return;
  }
  // output order among the selected: (rank, source index); the others sort last
  for (uint32_t i = threadIdx.x; i < n; i += NT) {
    const bool sel = pos[i] < m;
    const uint64_t r = (uint64_t)TR::rank(raw[i], dirmask);
    kh[i] = !sel ? ~0ull : (wide ? r : ((r << 32) | idx[i]));
    kl[i] = !sel ? ~0ull : (uint64_t)idx[i];
  }
  __syncthreads();
  count_ranks<NT, EC>(kh, wide ? kl : nullptr, n, pos);
  for (uint32_t i = threadIdx.x; i < n; i += NT) {
    const uint32_t p = pos[i];
    if (p < m) {
      out_keys[p] = raw[i];
      if (vals)
        vals.put(p, idx[i]);
    }
  }
}

// Sort the m items (raw[i], idx[i]) (i < m) by (rank, source index), the
// stable_sorted order of "Top-K: Determinism, Tie-Breaking, and Output
// Ordering" (Output ordering table), and write them to the output slots of
// one segment: a register bitonic sort of EPT elements per thread (items
// padded with keys that sort last); sort_and_write below picks it for up to
// one item per thread. Ranks up to 32 bits sort as one 64-bit
// composite rank<<32 | index with the item's slot beside it; 64-bit ranks as
// (rank, index<<32 | slot). `scratch` holds sort_scratch_bytes(m) bytes; the
// items must be visible to the whole block.
template <class TR, int NT, int EPT>
__device__ __forceinline__ void sort_write_ept(const typename TR::Raw* raw, const uint32_t* idx, uint32_t m,
                                               typename TR::Rank dirmask, unsigned char* scratch,
                                               typename TR::Raw* out_keys, const ValueSink& vals)
{
  uint64_t a[EPT], b[EPT];
#pragma unroll
  for (int r = 0; r < EPT; ++r) {
    const uint32_t e = threadIdx.x * (uint32_t)EPT + (uint32_t)r;
    a[r] = ~0ull;
    b[r] = ~0ull;
    if (e < m) {
      const uint64_t rk = (uint64_t)TR::rank(raw[e], dirmask);
      if constexpr (TR::kRankBits <= 32) {
        a[r] = (rk << 32) | idx[e];
        b[r] = e;
      } else {
        a[r] = rk;
        b[r] = ((uint64_t)idx[e] << 32) | e;
      }
    }
  }
  uint64_t* s1 = reinterpret_cast<uint64_t*>(scratch);
  uint64_t* s2 = s1 + (uint32_t)EPT * NT;
  reg_bitonic_sort<NT, EPT>(a, b, s1, s2);
#pragma unroll
  for (int r = 0; r < EPT; ++r) {
    const uint32_t e = threadIdx.x * (uint32_t)EPT + (uint32_t)r;
    if (e < m) {
      const uint32_t slot = (uint32_t)b[r];
      out_keys[e] = raw[slot];
      if (vals)
        vals.put(e, idx[slot]);
    }
  }
}

template <class TR, int NT>
__device__ __forceinline__ void sort_and_write(const typename TR::Raw* raw, const uint32_t* idx, uint32_t m,
                                               typename TR::Rank dirmask, unsigned char* scratch,
                                               typename TR::Raw* out_keys, const ValueSink& vals,
                                               bool stable = true)
{
  static_assert(NT == (int)kSortLanes, "sort scratch is sized for kSortLanes threads");
  const uint32_t n2 = next_pow2(m < 2 ? 2 : m);
  if (n2 <= (uint32_t)NT) {
    // one item per thread: registers and shuffles (measured faster up to 256
    // items; above, the shared-memory network below is)
    sort_write_ept<TR, NT, 1>(raw, idx, m, dirmask, scratch, out_keys, vals);
    return;
  }
  if constexpr (TR::kRankBits <= 32) {
    uint64_t* key = reinterpret_cast<uint64_t*>(scratch);
    uint32_t* pay = reinterpret_cast<uint32_t*>(key + n2);
    for (uint32_t i = threadIdx.x; i < n2; i += NT) {
      key[i] = i < m ? (((uint64_t)TR::rank(raw[i], dirmask) << 32) | idx[i]) : ~0ull;
      pay[i] = i;
    }
    __syncthreads();
    bitonic_sort_u64<NT>(key, pay, n2);
    for (uint32_t j = threadIdx.x; j < m; j += NT) {
      const uint32_t s = pay[j];
      out_keys[j] = raw[s];
      if (vals)
        vals.put(j, idx[s]);
    }
  } else if (!stable) {
    // sorted but not stable (equal keys in any order): 64-bit ranks sort on
    // the rank alone, the item's slot as payload
    uint64_t* key = reinterpret_cast<uint64_t*>(scratch);
    uint32_t* pay = reinterpret_cast<uint32_t*>(key + n2);
    for (uint32_t i = threadIdx.x; i < n2; i += NT) {
      key[i] = i < m ? (uint64_t)TR::rank(raw[i], dirmask) : ~0ull;
      pay[i] = i;
    }
    __syncthreads();
    bitonic_sort_u64<NT>(key, pay, n2);
    for (uint32_t j = threadIdx.x; j < m; j += NT) {
      const uint32_t s = pay[j];
      out_keys[j] = raw[s];
      if (vals)
        vals.put(j, idx[s]);
    }
  } else {
    uint64_t* khi = reinterpret_cast<uint64_t*>(scratch);
    uint64_t* klo = khi + n2;
    for (uint32_t i = threadIdx.x; i < n2; i += NT) {
      khi[i] = i < m ? (uint64_t)TR::rank(raw[i], dirmask) : ~0ull;
      klo[i] = i < m ? (((uint64_t)idx[i] << 32) | i) : ~0ull;
    }
    __syncthreads();
    bitonic_sort_u128<NT>(khi, klo, n2);
    for (uint32_t j = threadIdx.x; j < m; j += NT) {
      const uint32_t s = (uint32_t)klo[j];
      out_keys[j] = raw[s];
      if (vals)
        vals.put(j, idx[s]);
    }
  }
}

} // namespace segtopk
