// Block-level building blocks of the per-segment selection:
//   * radix digit selection over a candidate list held in shared memory,
//   * index-ordered compaction of the selected entries (warp ballots + a
//     block prefix scan), and
//   * a bitonic sort of the selected items for sorted output.
//
// The list is a structure of arrays in shared memory: raw key bits and the
// segment-local source index of every entry. Entries are kept in preference
// order: ascending source index for prefer_smaller_index (and unspecified),
// descending for prefer_larger_index. Among equal keys an earlier entry is
// therefore always the preferred one.
#pragma once

#include "common.cuh"

namespace segtopk {

constexpr int kDigitBits = 8;
constexpr int kBuckets = 1 << kDigitBits;

// Control block at the start of dynamic shared memory. Every CTA of a cluster
// has the same layout, so a field can be addressed in a peer through DSMEM.
struct Ctrl {
  uint64_t bars[8];            // one mbarrier per ring stage
  uint64_t scan_tot[2][32];    // per-warp packed totals of the block scans (double buffered)
  uint32_t hist[2][kBuckets];  // digit histograms (double buffered; zero outside a selection)
  uint32_t hist_merged[kBuckets]; // cluster leader: histogram pushed by the other CTAs
  uint32_t res[4];             // selection result of a pass: bucket, count before, bucket count
  uint32_t front_base;         // cross-CTA scan: selected entries of preceding CTAs
  uint32_t tie_base;           // cross-CTA scan: boundary ties of preceding CTAs
  uint32_t counts[2];          // this CTA's (front, tie) totals
  uint64_t red[32];            // block reductions
};
constexpr uint32_t kCtrlBytes = (sizeof(Ctrl) + 127u) & ~127u;

// Result of a radix selection: the k best entries are those with
// (rank & mask) < prefix ("front", strictly better than every boundary
// candidate) plus the first `ties` entries (in list order) with
// (rank & mask) == prefix. `mask` covers the resolved leading digits; it is
// all ones unless the selection stopped early because the boundary bucket
// held exactly the remaining count.
template <typename Rank>
struct Selection {
  Rank prefix;
  Rank mask;
  uint32_t ties;
};

// Warp 0 of the block: find the bucket holding the krem-th best candidate.
// `h` gives the 8 bucket counts this lane owns (buckets 8*lane .. 8*lane+7).
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

// Histogram of one digit over the list entries whose resolved digits match.
template <class TR, int NT>
__device__ __forceinline__ void build_hist(const typename TR::Raw* raw, uint32_t count,
                                           typename TR::Rank dirmask, typename TR::Rank prefix,
                                           typename TR::Rank mask, int shift, uint32_t* h)
{
  using Rank = typename TR::Rank;
  for (uint32_t e = threadIdx.x; e < count; e += NT) {
    const Rank r = TR::rank(raw[e], dirmask);
    if ((r & mask) == prefix)
      atomicAdd(&h[(uint32_t)(r >> shift) & (kBuckets - 1)], 1u);
  }
}

// Radix selection of the kk best of the first `count` list entries
// (count > kk > 0) inside one CTA: most-significant digit first, each pass
// histograms the digit over the candidates, finds the bucket holding the
// kk-th entry, narrows kk to that bucket and folds the digit into the
// prefix; it stops early when that bucket holds exactly the remaining count
// ("Implement Segmented TopK using Thread-Block-Clusters", sections 1.2
// "Radix (digit) top-k" and 1.4 "Early stop").
template <class TR, int NT>
__device__ Selection<typename TR::Rank> block_select(Ctrl& ctl, const typename TR::Raw* raw,
                                                     uint32_t count, uint32_t kk,
                                                     typename TR::Rank dirmask)
{
  using Rank = typename TR::Rank;
  constexpr int RB = TR::kRankBits;
  constexpr int P = RB / kDigitBits;
  Rank prefix = 0, mask = 0;
  uint32_t krem = kk;
  int p = 0;
  for (; p < P; ++p) {
    const int shift = RB - kDigitBits * (p + 1);
    build_hist<TR, NT>(raw, count, dirmask, prefix, mask, shift, ctl.hist[p & 1]);
    if (threadIdx.x < kBuckets)
      ctl.hist[(p + 1) & 1][threadIdx.x] = 0;
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        h[i] = ctl.hist[p & 1][8 * threadIdx.x + i];
      find_bucket(h, krem, ctl.res);
    }
    __syncthreads();
    const uint32_t b = ctl.res[0], before = ctl.res[1], cnt = ctl.res[2];
    krem -= before;
    prefix |= (Rank)b << shift;
    mask |= (Rank)(kBuckets - 1) << shift;
    if (cnt == krem)
      break;
  }
  if (p == P)
    p = P - 1;
  // restore the "both histograms zero" invariant (warp 0 read this one before the last barrier)
  if (threadIdx.x < kBuckets)
    ctl.hist[p & 1][threadIdx.x] = 0;
  Selection<Rank> s;
  s.prefix = prefix;
  s.mask = mask;
  s.ties = krem;
  return s;
}

// Walks the first `count` list entries in list order and classifies each as
// front ((rank & mask) < prefix), tie ((rank & mask) == prefix) or neither.
// For every front or tie entry it calls
//   sink(e, raw, idx, rank, is_front, front_rank, tie_rank)
// where front_rank / tie_rank count the front / tie entries before e in list
// order (warp ballots inside a warp's contiguous run of 128 entries, a block
// scan across warps). Returns the (front, tie) totals in every thread.
// The sink runs after a barrier that follows every thread's reads of the
// current tile, so it may overwrite list slots at or before the tile.
template <class TR, int NT, class Sink>
__device__ uint2 scan_list(Ctrl& ctl, const typename TR::Raw* raw, const uint32_t* idx,
                           uint32_t count, typename TR::Rank dirmask, typename TR::Rank prefix,
                           typename TR::Rank mask, Sink&& sink)
{
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  constexpr int NW = NT / 32;
  constexpr int R = 4; // rounds of 32 entries per warp and tile
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  uint32_t fronts_seen = 0, ties_seen = 0;
  int buf = 0;
  for (uint32_t tile = 0; tile < count; tile += NT * R) {
    Raw kr[R];
    uint32_t ki[R];
    Rank rk[R];
    uint32_t bf[R], bt[R];
    uint32_t wf = 0, wt = 0;
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const uint32_t e = tile + warp * (32 * R) + q * 32 + lane;
      const bool valid = e < count;
      kr[q] = valid ? raw[e] : Raw(0);
      ki[q] = valid ? idx[e] : 0u;
      rk[q] = TR::rank(kr[q], dirmask);
      const Rank mr = rk[q] & mask;
      bf[q] = __ballot_sync(kFull, valid && mr < prefix);
      bt[q] = __ballot_sync(kFull, valid && mr == prefix);
      wf += __popc(bf[q]);
      wt += __popc(bt[q]);
    }
    if (lane == 0)
      ctl.scan_tot[buf][warp] = (uint64_t)wf | ((uint64_t)wt << 32);
    __syncthreads();
    uint32_t fb = fronts_seen, tb = ties_seen, tf = 0, tt = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint64_t v = ctl.scan_tot[buf][w];
      if (w < (int)warp) {
        fb += (uint32_t)v;
        tb += (uint32_t)(v >> 32);
      }
      tf += (uint32_t)v;
      tt += (uint32_t)(v >> 32);
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const uint32_t fr = fb + __popc(bf[q] & lt);
      const uint32_t tr = tb + __popc(bt[q] & lt);
      const bool isf = (bf[q] >> lane) & 1u;
      const bool ist = (bt[q] >> lane) & 1u;
      if (isf || ist)
        sink(tile + warp * (32 * R) + q * 32 + lane, kr[q], ki[q], rk[q], isf, fr, tr);
      fb += __popc(bf[q]);
      tb += __popc(bt[q]);
    }
    fronts_seen += tf;
    ties_seen += tt;
    buf ^= 1;
  }
  return make_uint2(fronts_seen, ties_seen);
}

// Block-wide maximum of a rank value (every thread gets the result).
template <class Rank, int NT>
__device__ __forceinline__ Rank block_max(Ctrl& ctl, Rank v)
{
  v = warp_max(v);
  __syncthreads(); // ctl.red may still be read by a previous reduction
  if (lane_id() == 0)
    ctl.red[threadIdx.x >> 5] = (uint64_t)v;
  __syncthreads();
  Rank m = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const Rank x = (Rank)ctl.red[w];
    m = x > m ? x : m;
  }
  return m;
}

// In-place trim of the list to its kk best entries, keeping list order.
// Returns the largest rank kept (the new acceptance bound).
template <class TR, int NT>
__device__ __noinline__ typename TR::Rank trim_list(Ctrl& ctl, typename TR::Raw* raw, uint32_t* idx,
                                       uint32_t count, uint32_t kk, typename TR::Rank dirmask)
{
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  const Selection<Rank> s = block_select<TR, NT>(ctl, raw, count, kk, dirmask);
  Rank mx = 0;
  const uint32_t ties = s.ties;
  scan_list<TR, NT>(ctl, raw, idx, count, dirmask, s.prefix, s.mask,
                    [&](uint32_t, Raw kr, uint32_t ki, Rank rk, bool isf, uint32_t fr, uint32_t tr) {
                      if (isf || tr < ties) {
                        const uint32_t pos = fr + (tr < ties ? tr : ties);
                        raw[pos] = kr;
                        idx[pos] = ki;
                        mx = rk > mx ? rk : mx;
                      }
                    });
  return block_max<Rank, NT>(ctl, mx); // its barriers also publish the compacted list
}

// ---------------------------------------------------------------------------
// Bitonic sort of up to 2048 selected items by (rank ascending, source index
// ascending), the stable_sorted order of "Top-K: Determinism, Tie-Breaking,
// and Output Ordering" (Output ordering table). Keys are 64-bit composites
// rank<<32 | index for ranks up to 32 bits; 64-bit ranks use a (rank, index)
// pair. The payload is the item's slot in the source arrays.
// ---------------------------------------------------------------------------
template <int NT>
__device__ void bitonic_sort_u64(uint64_t* key, uint32_t* pay, uint32_t n2)
{
  for (uint32_t size = 2; size <= n2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < (n2 >> 1); i += NT) {
        const uint32_t lo = (i / stride) * 2 * stride + (i % stride);
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
      __syncthreads();
    }
  }
}

template <int NT>
__device__ void bitonic_sort_u128(uint64_t* khi, uint64_t* klo, uint32_t n2)
{
  for (uint32_t size = 2; size <= n2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = threadIdx.x; i < (n2 >> 1); i += NT) {
        const uint32_t lo = (i / stride) * 2 * stride + (i % stride);
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
      __syncthreads();
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
  return rank_bits > 32 ? n2 * 16u : n2 * 12u;
}

// Sort the m items (raw[i], idx[i]) (i < m) and write them to the output
// slots of one segment. `scratch` must hold sort_scratch_bytes(m) bytes.
template <class TR, int NT>
__device__ __noinline__ void sort_and_write(const typename TR::Raw* raw, const uint32_t* idx, uint32_t m,
                               typename TR::Rank dirmask, unsigned char* scratch,
                               typename TR::Raw* out_keys, int32_t* out_values,
                               const int32_t* values)
{
  using Rank = typename TR::Rank;
  const uint32_t n2 = next_pow2(m < 2 ? 2 : m);
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
      if (out_values)
        out_values[j] = values[idx[s]];
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
      if (out_values)
        out_values[j] = values[idx[s]];
    }
  }
}

} // namespace segtopk
