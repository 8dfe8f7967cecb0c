// Short segments with k <= 32: one warp, or a team of eight warps, per segment.
//
// A short segment does not need a CTA's streaming ring, digit passes and
// block barriers: one warp reads it straight from global memory and keeps its
// k best keys (k <= 32) in registers, one entry per lane, sorted (a team
// splits the segment between its warps and merges their lists). This is the
// small-segment path of "Implement Segmented TopK using Thread-Block-Clusters"
// (section 3.4 "Single-CTA path" and the launch classification of section
// 3.3: segments too small for a cluster are served by a smaller unit).
//
// Selection key. Every key becomes the composite (rank, preference index):
// the order-preserving rank code of the key (smaller = better) and the
// segment-local source index, inverted when larger indices are preferred.
// Composites are unique within a segment, so "the k smallest composites" is
// exactly the selection the contract of "Top-K: Determinism, Tie-Breaking,
// and Output Ordering" fixes ("Which items are selected?"), whatever order
// the keys are read in, with boundary ties taken by source index.
//
// Per warp: the sorted top list (lane i holds the i-th best composite) and
// a queue of up to 32 candidates in shared memory. A key is a candidate when
// its composite beats the current k-th entry; when the queue is full it is
// sorted (bitonic network over the lanes) and merged into the top list
// (lane i takes the better of top[i] and queue[31 - i], the 32 best of both
// in bitonic order, then a bitonic merge), which also tightens the k-th
// entry. Empty slots hold the all-ones composite; the only key that could
// share it (rank all ones and source index 0 with larger indices preferred)
// never beats it, and an empty slot decodes to that very key, so a segment
// shorter than k is still written exactly.
//
// Output: the first min(k, n) entries in composite order, which is the
// stable sorted order (rank, then source index) when smaller indices are
// preferred; with larger indices preferred the entries are re-sorted by
// (rank, source index) for stable sorted output (for sorted output without
// stability, composite order -- equal keys by descending index -- is kept). Key bits are read back from the
// segment by source index (so -0.0 keeps its sign), values likewise.
#pragma once

#include "stream_topk.cuh"

namespace segtopk {

constexpr int kWarpPathMaxK = 32;
// Warps per segment: one for short segments (a CTA of one warp, so that no
// warp waits for a sibling with a longer segment; up to 32 share an SM), a
// team of eight for longer ones.
constexpr int kWarpTeam = 8;

// Composite (rank, preference index); smaller is better.
template <class Rank, bool WIDE = (sizeof(Rank) == 8)>
struct Comp {
  uint64_t c; // rank << 32 | preference index (ranks of at most 32 bits)
  __device__ __forceinline__ static Comp make(Rank r, uint32_t pref) { return Comp{((uint64_t)r << 32) | pref}; }
  __device__ __forceinline__ static Comp worst() { return Comp{~0ull}; }
  __device__ __forceinline__ bool less(const Comp& o) const { return c < o.c; }
  __device__ __forceinline__ Comp xor_lane(int m) const { return Comp{__shfl_xor_sync(kFull, c, m)}; }
  __device__ __forceinline__ Comp from_lane(int src) const { return Comp{__shfl_sync(kFull, c, src)}; }
  __device__ __forceinline__ uint32_t pref() const { return (uint32_t)c; }
  __device__ __forceinline__ Rank rank() const { return (Rank)(c >> 32); }
};
template <class Rank>
struct Comp<Rank, true> {
  uint64_t r; // 64-bit rank
  uint32_t p; // preference index
  __device__ __forceinline__ static Comp make(Rank rr, uint32_t pref) { return Comp{(uint64_t)rr, pref}; }
  __device__ __forceinline__ static Comp worst() { return Comp{~0ull, ~0u}; }
  __device__ __forceinline__ bool less(const Comp& o) const { return r < o.r || (r == o.r && p < o.p); }
  __device__ __forceinline__ Comp xor_lane(int m) const
  {
    return Comp{__shfl_xor_sync(kFull, r, m), __shfl_xor_sync(kFull, p, m)};
  }
  __device__ __forceinline__ Comp from_lane(int src) const
  {
    return Comp{__shfl_sync(kFull, r, src), __shfl_sync(kFull, p, src)};
  }
  __device__ __forceinline__ uint32_t pref() const { return p; }
  __device__ __forceinline__ Rank rank() const { return (Rank)r; }
};

// One compare-exchange step of a bitonic network over the 32 lanes: the lane
// with the lower index of the pair keeps the smaller entry when `ascending`.
template <class E>
__device__ __forceinline__ E lane_exchange(E x, int stride, bool ascending)
{
  const E y = x.xor_lane(stride);
  const bool lower = (lane_id() & (uint32_t)stride) == 0;
  const bool take = (lower == ascending) ? y.less(x) : x.less(y);
  return take ? y : x;
}

// Sorts one entry per lane ascending over the warp (lane 0 the smallest).
template <class E>
__device__ __forceinline__ E warp_sort32(E x)
{
  const uint32_t lane = lane_id();
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
      x = lane_exchange(x, stride, (lane & (uint32_t)size) == 0 || size == 32);
  }
  return x;
}

// top and q sorted ascending over the lanes: the 32 smallest of both, sorted.
template <class E>
__device__ __forceinline__ E warp_merge32(E top, E q)
{
  const E rev = q.from_lane(31 - (int)lane_id());
  E m = rev.less(top) ? rev : top; // bitonic: top ascending, reversed queue descending
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1)
    m = lane_exchange(m, stride, true);
  return m;
}

// (rank, source index) of an entry, for the stable sorted output order.
template <class Rank>
struct OutKey {
  Rank r;
  uint32_t i;
  __device__ __forceinline__ bool less(const OutKey& o) const { return r < o.r || (r == o.r && i < o.i); }
  __device__ __forceinline__ OutKey xor_lane(int m) const
  {
    return OutKey{(Rank)__shfl_xor_sync(kFull, r, m), __shfl_xor_sync(kFull, i, m)};
  }
};

// One segment per CTA of W warps (W = 1 for short segments, 8 for longer
// ones), k <= 32, serving segments with n_lo < n <= n_hi. Warp w reads rounds
// w, w + W, ... of 32 * U 16-byte vectors and keeps its own top list. Its
// first round starts the list from the lanes' own best keys (sorted over the
// warp): the k-th of those k distinct keys already bounds the round, so the
// round does not queue every key while the list is empty. With
// W > 1 the warps share a bound: after each merge a warp lowers a shared word
// to its k-th entry (any warp's k-th entry bounds the segment's k-th: a key
// that does not beat it has k better keys), and every warp filters against
// the smaller of its own k-th entry and that word. At the end the W sorted
// lists are merged pairwise in shared memory.
template <KeyKind KK, int W>
__global__ void __launch_bounds__(32 * W, (W == 1) ? 32 : 4) warp_topk_kernel(const KernelParams p)
{
  using TR = KeyTraits<KK>;
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  using E = Comp<Rank>;
  constexpr bool kWide = sizeof(Rank) == 8;
  constexpr int VK = 16 / (int)sizeof(Raw); // keys per 16-byte vector
  constexpr int U = 4;                      // vectors per lane and round

  __shared__ E queue_all[W][32];             // candidate queues; at the end the warps' lists
  __shared__ uint4 stage_all[W][U][32];      // each lane's vectors of the current round
  __shared__ unsigned long long shared_bound; // W > 1: smallest k-th entry over the warps (its rank if wide)
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  E* queue = queue_all[warp];
  uint4 (*stage)[32] = stage_all[warp];

  const int64_t seg = (int64_t)blockIdx.x;
  if (seg >= p.num_segments)
    return;
  const int64_t g0 = p.offsets[seg];
  const int64_t g1 = p.offsets[seg + 1];
  const int64_t n64 = g1 > g0 ? g1 - g0 : 0;
  if (n64 <= p.n_lo)
    return; // uniform over the CTA
  if (n64 > p.n_hi) {
    if (p.flag_overlong && threadIdx.x == 0)
      raise_error(kErrSegmentTooLong);
    return;
  }
  const uint32_t n = (uint32_t)n64;
  const uint32_t k = (uint32_t)p.k;
  const uint32_t m = k < n ? k : n;
  const Rank dirmask = (Rank)p.dirmask;
  const bool is_max = dirmask != 0;
  const bool pl = p.prefer_larger != 0;
  const Raw* keys = reinterpret_cast<const Raw*>(p.keys);
  // 16-byte vectors are taken from the aligned address at or below keys[0];
  // in that vector array, key i of the key array is element i + lead
  const uintptr_t kaddr = reinterpret_cast<uintptr_t>(p.keys);
  const uint4* kvec = reinterpret_cast<const uint4*>(kaddr & ~(uintptr_t)15);
  const int64_t lead = (int64_t)((kaddr & 15u) / sizeof(Raw));
  const int64_t a0 = g0 + lead, a1 = g1 + lead; // the segment in vector-array elements
  if (W > 1) {
    if (threadIdx.x == 0)
      shared_bound = ~0ull;
    __syncthreads();
  }

  constexpr Rank kMaxRank = (TR::kRankBits == 64) ? ~(Rank)0 : (Rank)(((uint64_t)1 << TR::kRankBits) - 1);
  E top = E::worst();
  E thr = E::worst();   // the k-th entry of this warp's list
  uint64_t shb = ~0ull; // this warp's copy of shared_bound (W > 1)
  uint32_t qn = 0;      // queued candidates (warp-uniform)
  // Raw-domain prefilter of whole vectors: a key can enter only if its rank
  // is at most the bound's rank brank (bits braw; open: no such bound yet).
  bool open = true;
  Rank brank = 0;
  Raw braw = 0;

  // does composite c beat the k-th entry (and the shared bound)?
  auto beats = [&](const E& c) {
    if constexpr (kWide)
      return c.less(thr) && (W == 1 || c.rank() <= (Rank)shb);
    else
      return c.c < (W == 1 ? thr.c : min(thr.c, shb));
  };
  auto set_bound = [&]() {
    Rank tr = thr.rank();
    if (W > 1) {
      const Rank sr = kWide ? (Rank)shb : (Rank)(shb >> 32);
      tr = sr < tr ? sr : tr;
    }
    open = tr >= kMaxRank; // an empty slot, or a rank that admits every key
    if (!open) {
      brank = tr;
      braw = TR::unrank(tr, dirmask);
    }
  };
  auto refresh_shared = [&]() { // warp-uniform read of the shared bound
    if (W > 1) {
      uint64_t x = 0;
      if (lane == 0)
        x = *reinterpret_cast<volatile unsigned long long*>(&shared_bound);
      shb = __shfl_sync(kFull, x, 0);
      set_bound();
    }
  };
  auto flush = [&]() {
    __syncwarp();
    const E x = lane < qn ? queue[lane] : E::worst();
    top = warp_merge32(top, warp_sort32(x));
    thr = top.from_lane((int)k - 1);
    qn = 0;
    if (W > 1 && lane == 0) {
      if constexpr (kWide)
        atomicMin(&shared_bound, (unsigned long long)thr.rank());
      else
        atomicMin(&shared_bound, (unsigned long long)thr.c);
    }
    set_bound();
    __syncwarp(); // the queue is rewritten next
  };
  auto composite = [&](Raw key, uint32_t idx) { return E::make(TR::rank(key, dirmask), pl ? ~idx : idx); };

  // 16-byte vectors covering the segment. A vector is read whole when it ends
  // inside the segment (its start, if before the segment, is still inside
  // the aligned 16 bytes that hold the segment's first key); the last,
  // partial one key by key.
  const int64_t v_first = a0 / VK;
  const int64_t v_end = (a1 + VK - 1) / VK;
  bool first = true;
  for (int64_t vb = v_first + (int64_t)warp * 32 * U; vb < v_end; vb += (int64_t)32 * U * W) {
    uint4 vec[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = vb + u * 32 + lane;
      vec[u] = make_uint4(0, 0, 0, 0);
      if (v < v_end) {
        if ((v + 1) * VK <= a1) {
          vec[u] = __ldg(kvec + v);
        } else {
#pragma unroll
          for (int j = 0; j < VK; ++j) {
            const int64_t e = v * VK + j - lead; // key-array index
            if (e >= g0 && e < g1)
              vec_set_key<Raw>(vec[u], j, keys[e]);
          }
        }
      }
    }
    uint32_t taken = 0; // first round: the lane's own best key, already in the list
    if (first) {
      first = false;
      E best = E::worst();
      int best_s = -1;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t rel = (vb + u * 32 + lane) * VK - a0;
#pragma unroll
        for (int j = 0; j < VK; ++j) {
          if (rel + j >= 0 && rel + j < (int64_t)n) {
            const E c = composite(vec_key<Raw>(vec[u], j), (uint32_t)(rel + j));
            if (c.less(best)) {
              best = c;
              best_s = u * VK + j;
            }
          }
        }
      }
      top = warp_sort32(best); // lanes without a key offer an empty slot
      thr = top.from_lane((int)k - 1);
      if (W > 1 && lane == 0) {
        if constexpr (kWide)
          atomicMin(&shared_bound, (unsigned long long)thr.rank());
        else
          atomicMin(&shared_bound, (unsigned long long)thr.c);
      }
      set_bound();
      taken = best_s >= 0 ? 1u << best_s : 0u;
    }
    refresh_shared();
    // this lane's keys that beat the bound (bit u * VK + j); keys j of
    // vector v belong to the segment for lo <= j < hi
    uint32_t cand = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = vb + u * 32 + lane;
      const int64_t rel = v * VK - a0; // segment index of key 0 of the vector
      const int lo = rel < 0 ? (int)-rel : 0;
      const int64_t rest = (int64_t)n - rel; // keys of the segment from key 0 of the vector on
      const int hi = rest < VK ? (int)rest : VK;
      stage[u][lane] = vec[u];
      if (hi > lo && (open || TR::may_pass(vec[u], braw, brank, is_max, false))) {
#pragma unroll
        for (int j = 0; j < VK; ++j) {
          if (j >= lo && j < hi && beats(composite(vec_key<Raw>(vec[u], j), (uint32_t)(rel + j))))
            cand |= 1u << (u * VK + j);
        }
      }
    }
    cand &= ~taken;
    // queue them, one per lane at a time (re-read from the lane's stage; the
    // bound may have tightened since), merging whenever the queue fills
    while (__any_sync(kFull, cand != 0)) {
      bool enter = false;
      E c = E::worst();
      if (cand) {
        const int s = __ffs(cand) - 1;
        cand &= cand - 1;
        const int u = s / VK, j = s % VK;
        const Raw key = reinterpret_cast<const Raw*>(&stage[u][lane])[j];
        c = composite(key, (uint32_t)((vb + u * 32 + lane) * VK + j - a0));
        enter = beats(c);
      }
      uint32_t mask = __ballot_sync(kFull, enter);
      if (qn + __popc(mask) > 32u) {
        flush();
        enter = enter && beats(c);
        mask = __ballot_sync(kFull, enter);
      }
      if (enter)
        queue[qn + __popc(mask & lanemask_lt())] = c;
      qn += __popc(mask);
    }
  }
  if (qn)
    flush();

  if (W > 1) {
    // merge the warps' sorted lists pairwise (the queues are free now)
    queue[lane] = top;
    __syncthreads();
#pragma unroll
    for (int step = W / 2; step > 0; step >>= 1) {
      if ((int)warp < step) {
        const E r = warp_merge32(queue_all[warp][lane], queue_all[warp + step][lane]);
        __syncwarp();
        queue_all[warp][lane] = r;
      }
      __syncthreads();
    }
    if (warp != 0)
      return;
    top = queue_all[0][lane];
  }

  // lanes [0, m) hold the selection in composite order
  uint32_t idx = pl ? ~top.pref() : top.pref();
  if (p.sorted && pl && p.stable) { // (for sorted, not stable, composite order is a valid order)
    OutKey<Rank> o{lane < m ? top.rank() : ~(Rank)0, lane < m ? idx : ~0u};
    o = warp_sort32(o);
    idx = o.i;
  }
  if (lane < m) {
    Raw* out_keys = reinterpret_cast<Raw*>(p.out_keys) + seg * (int64_t)k;
    out_keys[lane] = keys[g0 + idx];
    if (p.out_values) {
      const int64_t vb = p.value_bytes;
      const ValueSink vals{static_cast<char*>(p.out_values) + seg * (int64_t)k * vb,
                           p.values ? static_cast<const char*>(p.values) + g0 * vb : nullptr, vb == 8 ? 1 : 0};
      vals.put(lane, idx);
    }
  }
}

} // namespace segtopk
