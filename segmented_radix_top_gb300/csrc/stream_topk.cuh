// The segment kernel: one CTA, or one thread-block cluster, per segment.
//
// Method ("Implement Segmented TopK using Thread-Block-Clusters", sections
// 1.2 - 1.6 and 2): multi-pass radix digit selection with a final filter that
// writes the keys strictly beyond the splitter plus exactly enough boundary
// ties, ties taken in source-index order.
//
// GB300 design (what differs from the pages' CUB kernel):
//  * Keys stream once from HBM through a ring of 32 KiB shared-memory stages
//    filled by 1-D bulk copies (TMA), one mbarrier per stage, chunks visited
//    in preference order (descending source index for prefer_larger_index).
//  * Instead of keeping the whole segment resident and re-reading it every
//    pass, each CTA keeps a bounded candidate list in shared memory that
//    always contains the best k keys it has read so far. A key enters the
//    list only if it ranks below the current bound (the rank of the k-th
//    best key kept); a one-compare-per-key filter in the key's own domain
//    rejects almost every key before its rank is computed. When the list
//    could overflow, it is trimmed back to k entries by the radix digit
//    selection, which also tightens the bound. Keys arriving after a trim
//    come later in preference order than every kept key, so a key that only
//    ties the bound is rightly rejected.
//  * A cluster of C CTAs splits a long segment into C contiguous slices.
//    When the C local top-k lists fit in one CTA, they are gathered into the
//    leader through DSMEM (one cluster barrier) and the leader selects from
//    them. Otherwise the pages' cluster merge runs: per-CTA digit histograms
//    folded into the leader through DSMEM, the leader's scan broadcast back,
//    a cross-CTA count scan of (front, tie) counts in preference order, each
//    CTA picking its share of the boundary ties by source index, and for
//    sorted output a DSMEM gather of the selected items into the leader.
#pragma once

#include "block_select.cuh"

namespace segtopk {

// Threads per CTA.
constexpr int kCtaThreads = 256;

// A kernel profile: CTAs an SM is sized for, 16-byte vectors a thread filters
// per ring stage (a stage holds kCtaThreads * VEC_PER_THREAD vectors), the
// capacity of the selection's candidate-position buffer, and the ring's
// stages (a power of two, so that stage and phase are bit operations).
template <int CTAS_PER_SM, int VEC_PER_THREAD, uint32_t CAND_CAP, uint32_t STAGES = 2>
struct CtaProfile {
  static constexpr int kCtasPerSm = CTAS_PER_SM;
  static constexpr int kVecPerThread = VEC_PER_THREAD;
  static constexpr uint32_t kChunkBytes = 16u * (uint32_t)VEC_PER_THREAD * (uint32_t)kCtaThreads;
  static constexpr uint32_t kCandCap = CAND_CAP;
  static constexpr uint32_t kCandBytes = CAND_CAP * 2u;
  static constexpr uint32_t kStages = STAGES;
  static constexpr uint32_t kRingBytes = STAGES * kChunkBytes;
  static_assert(STAGES >= 2 && STAGES <= 8 && (STAGES & (STAGES - 1)) == 0, "ring stages");
};
// Long segments served by one wave of CTAs or clusters: two CTAs per SM,
// 32 KiB stages (fewer, larger chunks per segment).
using ProfileLong = CtaProfile<2, 8, 4096>;
// Several waves of single-CTA segments: three CTAs per SM, 16 KiB stages,
// so that one CTA's selections overlap the others' streams.
using ProfileMany = CtaProfile<3, 4, 2048>;

struct KernelParams {
  const void* keys;
  const void* values;    // int32 or int64 payload (value_bytes), or null
  const int64_t* offsets;
  void* out_keys;
  void* out_values;
  int64_t num_segments;
  int64_t n_lo;          // this launch serves segments with n_lo < n <= n_hi
  int64_t n_hi;
  uint64_t dirmask;      // rank = T(key) ^ dirmask: all ones for max, zero for min
  int32_t k;
  uint32_t list_cap;     // candidate list capacity (entries)
  uint32_t ring_bytes;   // ring region bytes (also sort / gather scratch)
  int32_t prefer_larger; // tie preference: larger source index first
  int32_t sorted;        // write the selected items in stable sorted order
  int32_t merge_gather;  // cluster merge: 2 gather whole lists, 1 gather local top-k, 0 histograms
  int32_t flag_overlong; // report segments longer than n_hi
  uint32_t spec_keys;    // sample size of the speculative first bound
  float spec_z;          // its margin: mu + spec_z * sqrt(mu) + spec_c sample keys are kept
  float spec_c;
  int32_t spec_small;    // small targets by warp minimums (exact) rather than digit passes (slack stop)
  long long wait_limit;  // clock cycles after which a wait on a bulk copy gives up
  int32_t value_bytes;   // 4 or 8
  int32_t tie_any;       // not_guaranteed: surplus boundary ties may be taken in any order
  int32_t stable;        // sorted output keeps equal keys in source-index order
  uint32_t test_extra_tx; // instrumented build only: bytes added to a slice's first copy's expected count
};

// Per-CTA counters of the statistics build, flushed once per CTA.
static __device__ unsigned long long g_stats[kStatCount];


// Host and device agree on the dynamic shared-memory layout.
__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }
__host__ __device__ inline uint32_t list_bytes(uint32_t cap, uint32_t key_bytes)
{
  return align16(cap * key_bytes) + cap * 4u;
}
// Least sample of an exact first bound (keys of the first chunk; at least
// four times k are taken).
constexpr uint32_t kBootKeys = 2048;

template <KeyKind KK, int NT, class PR>
__global__ void __launch_bounds__(NT, PR::kCtasPerSm) stream_topk_kernel(const KernelParams p)
{
  using TR = KeyTraits<KK>;
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  constexpr int VK = 16 / (int)sizeof(Raw);     // keys per 16-byte vector
  constexpr uint32_t kChunkBytes = PR::kChunkBytes;
  constexpr uint32_t kCandCap = PR::kCandCap; // candidate positions a selection keeps between passes
  constexpr int U = (int)kChunkBytes / 16 / NT; // vectors per thread per chunk
  constexpr uint32_t kChunkVec = kChunkBytes / 16;
  static_assert(U >= 1 && U <= 8, "chunk / thread configuration");
  static_assert(kChunkBytes / sizeof(Raw) >= NT, "a chunk gives every thread keys");

  extern __shared__ __align__(128) unsigned char smem[];
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem);
  unsigned char* ring = smem + kCtrlBytes;
  // two candidate-list buffers: a trim writes the kept entries into the spare one
  unsigned char* lists = ring + p.ring_bytes;
  const uint32_t lbytes = list_bytes(p.list_cap, sizeof(Raw));
  Raw* list_raw = reinterpret_cast<Raw*>(lists);
  uint32_t* list_idx = reinterpret_cast<uint32_t*>(lists + align16(p.list_cap * sizeof(Raw)));
  Raw* spare_raw = reinterpret_cast<Raw*>(lists + lbytes);
  uint32_t* spare_idx = reinterpret_cast<uint32_t*>(lists + lbytes + align16(p.list_cap * sizeof(Raw)));
  uint16_t* cand_pos = reinterpret_cast<uint16_t*>(lists + 2 * lbytes);
  const CandBuf cbuf{cand_pos, kCandCap, 0u};

  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int64_t seg = (C == 1) ? (int64_t)blockIdx.x : (int64_t)cluster_id_x();
  if (seg >= p.num_segments)
    return;
  const int64_t g0 = p.offsets[seg];
  const int64_t g1 = p.offsets[seg + 1];
  const int64_t n64 = g1 > g0 ? g1 - g0 : 0;
  if (n64 <= p.n_lo)
    return; // another launch serves this segment (the whole cluster returns)
  if (n64 > p.n_hi) {
    if (p.flag_overlong && threadIdx.x == 0 && rank == 0)
      raise_error(kErrSegmentTooLong);
    return;
  }
#ifdef SEGTOPK_STATS
  const long long t_start = clock64();
#endif
  const uint32_t n = (uint32_t)n64;
  const uint32_t k = (uint32_t)p.k;
  const uint32_t m = k < n ? k : n;
  const Rank dirmask = (Rank)p.dirmask;
  const bool is_max = dirmask != 0;
  const bool fwd = !p.prefer_larger;
  const bool tie_any = p.tie_any != 0;
  constexpr uint32_t S = PR::kStages;

  // ---- front-loaded shared-memory initialisation ----
  for (uint32_t i = threadIdx.x; i < kBuckets; i += NT) {
    ctl.hist_m0[i] = 0;
    ctl.hist_merged[i] = 0;
  }
  clear_slot<NT>(ctl.slot[0]);
  clear_slot<NT>(ctl.slot[1]);
  clear_slot<NT>(ctl.slot[2]);
  if (threadIdx.x == 0) {
    ctl.chunk_count[0] = ctl.chunk_count[1] = ctl.chunk_count[2] = 0;
    ctl.abort = 0;
#ifdef SEGTOPK_STATS
    for (int i = 0; i < kStatCount; ++i)
      ctl.stat[i] = 0;
#endif
    ctl.gather_count = 0;
    ctl.front_base = 0;
    ctl.tie_base = 0;
    for (uint32_t s = 0; s < S; ++s)
      mbar_init(&ctl.bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this CTA's slice of the segment ----
  // The body is the run of whole 16-byte vectors of the segment; the keys
  // before its first vector (head) and after its last (tail) are read one by
  // one. Any element-aligned key pointer works.
  const Raw* seg_keys = reinterpret_cast<const Raw*>(p.keys) + g0;
  const uint32_t mis = (uint32_t)((reinterpret_cast<uintptr_t>(seg_keys) & 15u) / sizeof(Raw));
  uint32_t head = (uint32_t)((VK - (int)mis) % VK); // unaligned leading keys
  if (head > n)
    head = n;
  const uint32_t body_v = (n - head) / VK;
  const uint32_t tail = n - head - body_v * VK; // unaligned trailing keys
  const uint32_t v_lo = (uint32_t)(((uint64_t)body_v * rank) / C);
  const uint32_t v_hi = (uint32_t)(((uint64_t)body_v * (rank + 1)) / C);
  const uint32_t nvec = v_hi - v_lo;
  const uint32_t nchunks = (nvec + kChunkVec - 1) / kChunkVec;
  const bool has_head = rank == 0 && head > 0;
  const bool has_tail = rank == C - 1 && tail > 0;
  SEGTOPK_STAT_ADD(kStatCtas, 1);

  auto chunk_of_step = [&](uint32_t s) { return fwd ? s : nchunks - 1 - s; };
  // ---- streaming selection state (uniform across the block) ----
  const uint32_t L = p.list_cap;
  const uint32_t n_slice = nvec * VK + (has_head ? head : 0u) + (has_tail ? tail : 0u);
  // a trim may keep up to this many entries beyond k (fewer digit passes)
  const uint32_t trim_slack = min((L - k) / 4u, max(k / 2u, 16u));
  uint32_t count = 0; // list entries
  bool open = true;   // no bound yet: every key is accepted
  Bound<Raw, Rank> bound{(Rank)0, (Raw)0};
  uint32_t step = 0;  // edges and chunks offered so far (selects the append counter)
  uint32_t sel_pass = 0; // digit-selection passes so far (selects the pass slot)
  const bool pl = p.prefer_larger != 0;

  auto set_bound = [&](Rank tau, uint32_t kept) {
    bound.tau = tau;
    bound.raw = TR::unrank(tau, dirmask);
    open = false;
    count = kept;
  };
  auto swap_lists = [&]() {
    Raw* tr = list_raw;
    list_raw = spare_raw;
    spare_raw = tr;
    uint32_t* ti = list_idx;
    list_idx = spare_idx;
    spare_idx = ti;
  };
  // Keep the k best of the list and `n_ext` keys at `ext` (indices idx0..)
  // -- with slack, up to k + slack entries that include them -- in the spare
  // buffer, which becomes the list.
  auto select_union = [&](const Raw* ext, uint32_t idx0, uint32_t n_ext, uint32_t slack) {
    const Kept<Rank> kp = trim_into<TR, NT>(ctl, sel_pass, Src<Raw>{list_raw, list_idx, count, ext, idx0, n_ext},
                                            spare_raw, spare_idx, k, slack, dirmask, pl, cbuf, tie_any);
    sel_pass = kp.pass;
    swap_lists();
    set_bound(kp.max_rank, kp.n);
  };
  auto trim_list = [&](uint32_t slack) {
    SEGTOPK_STAT_ADD(kStatTrims, 1);
    select_union(nullptr, 0u, 0u, slack);
  };

  // Test the flagged vectors exactly (bit j of mayv: vector j, with vc[j]
  // keys from slot 0 and source indices i0[j] + slot, may hold a key that
  // beats the bound) and append the accepted keys at list positions count +
  // (a per-lane atomic on this step's counter). Returns true if an append
  // would overflow the list (nothing is written for that lane then).
  auto append_flagged = [&](const uint4 (&vec)[U], const uint32_t (&vc)[U], const uint32_t (&i0)[U],
                            uint32_t mayv) {
    bool overflow = false;
    if (mayv) {
      uint32_t acc[U];
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        acc[j] = 0;
        if ((mayv >> j) & 1u) {
          const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
          for (int i = 0; i < VK; ++i)
            if ((uint32_t)i < vc[j] && (open || TR::rank(kv[i], dirmask) < bound.tau))
              acc[j] |= 1u << i;
          c += __popc(acc[j]);
        }
      }
      if (c) {
        const uint32_t pos = count + atomicAdd(&ctl.chunk_count[step % 3], c);
        if (pos + c > L) {
          overflow = true;
        } else {
          uint32_t w = pos;
#pragma unroll
          for (int j = 0; j < U; ++j) {
            if (acc[j]) {
              const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
              for (int i = 0; i < VK; ++i) {
                if ((acc[j] >> i) & 1u) {
                  list_raw[w] = kv[i];
                  list_idx[w] = i0[j] + (uint32_t)i;
                  ++w;
                }
              }
            }
          }
        }
      }
    }
    return overflow;
  };
  // Offer up to U loose vectors (the edges): every key when no bound is set yet.
  auto offer = [&](const uint4 (&vec)[U], const uint32_t (&vc)[U], const uint32_t (&i0)[U]) {
    uint32_t mayv = 0;
#pragma unroll
    for (int j = 0; j < U; ++j)
      if (vc[j] && (open || TR::may_pass(vec[j], bound.raw, bound.tau, is_max, true)))
        mayv |= 1u << j;
    return append_flagged(vec, vc, i0, mayv);
  };

  // After a step's barrier: account its appends (unless a selection replaced
  // the list) and recycle the counter of the step before, which every thread
  // read after the previous barrier; it is next used two steps from now.
  auto finish_step = [&](bool counted) {
    if (counted)
      count += ctl.chunk_count[step % 3];
    if (threadIdx.x == 0)
      ctl.chunk_count[(step + 2) % 3] = 0;
    ++step;
  };

  // Candidate bits of this thread's vectors [v0, v1) of a ring stage: bits
  // j * VK .. j * VK + VK - 1 hold TR::pass_bits of vector j = j * NT +
  // thread (a superset of the keys ranking below the bound: exact but for
  // NaNs and, for 64-bit keys, ties of the high words).
  using CandMask = typename std::conditional<(U * VK > 32), uint64_t, uint32_t>::type;
  auto candidate_bits = [&](const uint4* stage, uint32_t v0, uint32_t v1) {
    uint4 vv[U];
#pragma unroll
    for (int j = 0; j < U; ++j) // all loads first (vectors outside [v0, v1) are masked below)
      vv[j] = stage[(uint32_t)j * NT + threadIdx.x];
    CandMask m = 0;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t t = (uint32_t)j * NT + threadIdx.x;
      const uint32_t b = TR::pass_bits(vv[j], bound.raw, bound.tau, is_max);
      m |= (CandMask)((t >= v0 && t < v1) ? b : 0u) << (j * VK);
    }
    return m;
  };

  // Test this thread's candidates exactly (rank below the bound), each read
  // from the stage, and append the accepted ones at list positions count +
  // (an atomic on this step's counter, one per key). A lane loops over its
  // own candidates only, so a warp takes as many rounds as its busiest lane
  // has candidates. Returns true if an append would overflow the list
  // (that key is not written).
  auto append_candidates = [&](const Raw* stage_keys, CandMask m, uint32_t idx0) {
    bool overflow = false;
    while (m) {
      uint32_t q;
      if constexpr (sizeof(CandMask) == 8)
        q = (uint32_t)__ffsll((long long)m) - 1u;
      else
        q = (uint32_t)__ffs(m) - 1u;
      m &= m - 1u;
      const uint32_t j = q / (uint32_t)VK;
      const uint32_t e = (j * NT + threadIdx.x) * VK + TR::key_of_bit(q % (uint32_t)VK);
      const Raw key = stage_keys[e];
      if (TR::rank(key, dirmask) < bound.tau) {
        const uint32_t pos = count + atomicAdd(&ctl.chunk_count[step % 3], 1u);
        if (pos < L) {
          list_raw[pos] = key;
          list_idx[pos] = idx0 + e;
        } else {
          overflow = true;
        }
      }
    }
    return overflow;
  };

  // Vectors [v0, v1) of a ring stage: offer them; if the list overflows,
  // trim the list (as it was before the attempt) to tighten the bound and
  // offer them again; if they overflow even a trimmed list, keep the k best
  // of the list and all of those keys. Then the stage is released
  // (`release` refills it).
  auto process_vectors = [&](const uint4* stage, uint32_t v0, uint32_t v1, uint32_t idx0, auto&& release) {
    const Raw* stage_keys = reinterpret_cast<const Raw*>(stage);
    bool trimmed = false;
    for (;;) {
      const CandMask m = candidate_bits(stage, v0, v1);
      bool overflow = false;
      if (__any_sync(kFull, m != 0)) { // most warps hold no candidate
        SEGTOPK_STAT_ADD(kStatSlowChunks, 1);
        overflow = append_candidates(stage_keys, m, idx0);
      }
      if (!__syncthreads_or(overflow)) {
        finish_step(true);
        break;
      }
      finish_step(false); // drop this attempt's appends
      SEGTOPK_STAT_ADD(kStatFallbackChunks, 1);
      if (!trimmed && count > k) {
        trim_list(trim_slack);
        trimmed = true;
      } else {
        select_union(stage_keys + (size_t)v0 * VK, idx0 + v0 * VK, (v1 - v0) * VK, trim_slack);
        break;
      }
    }
    release();
  };

  // Unaligned head / tail keys: plain loads, one per thread.
  auto offer_edge = [&](uint32_t e_begin, uint32_t e_cnt) {
    if (count + e_cnt > L) // keep room for the edge (e_cnt < 8)
      trim_list(trim_slack);
    uint4 vec[U];
    uint32_t vc[U], i0[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      vec[j] = make_uint4(0, 0, 0, 0);
      vc[j] = 0;
      i0[j] = 0;
    }
    if (threadIdx.x < e_cnt) {
      reinterpret_cast<Raw*>(&vec[0])[0] = seg_keys[e_begin + threadIdx.x];
      vc[0] = 1;
      i0[0] = e_begin + threadIdx.x;
    }
    offer(vec, vc, i0); // cannot overflow: count + e_cnt <= L
    __syncthreads();
    finish_step(true);
  };

  // One pass over this CTA's slice: edges and chunks in preference order.
  // With allow_spec, the first bound may come from a sample (spec_into):
  // the sample's share of the slice's k best plus four standard deviations,
  // so that the list stays small and trims are rare. Returns whether that
  // speculative bound was used; the caller then checks that the slice gave
  // at least min(k, n_slice) entries.
  uint32_t gstep = 0; // ring steps over all passes (stage and mbarrier phase)
  auto stream_pass = [&](bool allow_spec) {
#ifdef SEGTOPK_STATS
    const long long t_pass = clock64();
#endif
    bool spec_used = false;
    const uint32_t gbase = gstep;
    uint32_t issued = 0; // thread 0: chunks issued in this pass
    uint32_t landed = 0; // thread 0: chunks 0 .. landed-1 seen complete
    auto issue_next = [&]() {
      const uint32_t g = gbase + issued;
      const uint32_t v0 = v_lo + chunk_of_step(issued) * kChunkVec;
      const uint32_t nv = min(kChunkVec, v_hi - v0);
      const uint32_t st = g % S;
      uint32_t extra = 0;
#ifdef SEGTOPK_TEST_HOOKS
      if (issued == 0)
        extra = p.test_extra_tx; // the wait on this copy then runs out (tests of the bounded wait)
#endif
      mbar_arrive_expect_tx(&ctl.bars[st], nv * 16u + extra);
      bulk_load(ring + (size_t)st * kChunkBytes, seg_keys + head + (size_t)v0 * VK, nv * 16u, &ctl.bars[st]);
      ++issued;
    };
    if (threadIdx.x == 0 && !ctl.abort) {
      while (issued < S && issued < nchunks)
        issue_next();
    }

    if (has_head && fwd)
      offer_edge(0, head);
    if (has_tail && !fwd)
      offer_edge(n - tail, tail);

    for (uint32_t s = 0; s < nchunks; ++s) {
      const uint32_t g = gbase + s;
      const uint32_t st = g % S;
      // Every thread waits (bounded) for the stage. A wait that gives up
      // sets the CTA's stop flag but changes no control flow: every thread
      // still runs every barrier below, on whatever the stage holds, no
      // further copy is issued, and the CTA writes no output.
      if (!*reinterpret_cast<volatile uint32_t*>(&ctl.abort)) {
#ifdef SEGTOPK_STATS
        const long long tw = clock64();
#endif
        if (!mbar_wait(&ctl.bars[st], (g / S) & 1u, p.wait_limit))
          atomicOr(&ctl.abort, 1u);
        else if (threadIdx.x == 0)
          landed = s + 1;
        SEGTOPK_STAT_ADD(kStatWaitCycles, clock64() - tw);
      }
      // refills this stage once every read of it is over (only after this
      // thread saw every copy so far land, and streaming goes on); once per chunk
      bool released = false;
      auto release = [&]() {
        if (!released && threadIdx.x == 0 && issued < nchunks && landed == s + 1 &&
            !*reinterpret_cast<volatile uint32_t*>(&ctl.abort))
          issue_next();
        released = true;
      };
      const uint32_t vb = v_lo + chunk_of_step(s) * kChunkVec;
      const uint32_t nv = min(kChunkVec, v_hi - vb);
      const uint4* stage = reinterpret_cast<const uint4*>(ring + (size_t)st * kChunkBytes);
      const Raw* stage_keys = reinterpret_cast<const Raw*>(stage);
      const uint32_t nkeys = nv * VK;
      const uint32_t idx0 = head + vb * VK;
      if (open) {
        if (count + nkeys <= k) {
          // still fewer than k keys in all: every one of them is selected so far
          for (uint32_t e = threadIdx.x; e < nkeys; e += NT) {
            list_raw[count + e] = stage_keys[e];
            list_idx[count + e] = idx0 + e;
          }
          __syncthreads();
          count += nkeys;
        } else {
#ifdef SEGTOPK_STATS
          const long long tb = clock64();
#endif
          // the first bound, from the list and the most preferred keys of this
          // chunk (the rest of the chunk comes later in preference order and
          // is offered against it): speculative from p.spec_keys of them, else
          // the exact k best of enough to pass k, at least kBootKeys
          uint32_t nb = 0;
          bool done = false;
          bool tie_block = false; // the speculative selection met a tie block at rank tie_rank
          Rank tie_rank = 0;
          if (allow_spec) {
            const uint32_t nbs = min(nv, (p.spec_keys + VK - 1) / VK);
            const uint32_t ns = count + nbs * VK;
            const float mu = (float)k * (float)ns / (float)n_slice;
            const uint32_t mm = (uint32_t)ceilf(mu + p.spec_z * sqrtf(mu) + p.spec_c);
            if (mm < k && mm < ns) {
              const uint32_t b0 = fwd ? 0u : nv - nbs;
              // a small target over ring keys only: warp minimums; else digit passes
              const Spec<Rank> sp =
                (p.spec_small && count == 0 && mm <= 32u && nbs * VK <= 8u * NT)
                  ? (nbs * VK <= 4u * NT
                       ? spec_small<TR, NT, 4>(ctl, sel_pass, stage_keys + (size_t)b0 * VK, idx0 + b0 * VK, nbs * VK,
                                               mm, spare_raw, spare_idx, L, dirmask,
                                               reinterpret_cast<uint32_t*>(cbuf.pos))
                       : spec_small<TR, NT, 8>(ctl, sel_pass, stage_keys + (size_t)b0 * VK, idx0 + b0 * VK, nbs * VK,
                                               mm, spare_raw, spare_idx, L, dirmask,
                                               reinterpret_cast<uint32_t*>(cbuf.pos)))
                  : spec_into<TR, NT>(ctl, sel_pass,
                                      Src<Raw>{list_raw, list_idx, count, stage_keys + (size_t)b0 * VK,
                                               idx0 + b0 * VK, nbs * VK},
                                      spare_raw, spare_idx, mm, L, dirmask, cbuf);
              sel_pass = sp.pass;
              tie_block = sp.tie_block;
              tie_rank = sp.edge;
              if (sp.ok) {
                swap_lists();
                set_bound(sp.edge + 1, sp.n); // accept rank <= edge
                spec_used = true;
                done = true;
                nb = nbs;
              }
            }
          }
          if (!done) {
            // several times k, so that the sample's k-th key sits where the
            // slice's will (with fewer, a tie block cut short by sampling
            // noise leaves the bound below the ties and lets them all in)
            const uint32_t want = max(k + 1 - count, max(4u * k, (uint32_t)kBootKeys));
            nb = min(nv, (want + VK - 1) / VK);
            const uint32_t b0 = fwd ? 0u : nv - nb;
            bool tied = false;
            if (tie_block && count == 0) {
              // the k-th key probably lies in the tie block just met: the keys
              // better than it and the first ties in preference order
              const Kept<Rank> kp =
                tie_block_into<TR, NT>(ctl, sel_pass, Src<Raw>{list_raw, list_idx, 0u, stage_keys + (size_t)b0 * VK,
                                                                idx0 + b0 * VK, nb * VK},
                                       tie_rank, k, spare_raw, spare_idx, L, dirmask, pl);
              if (kp.n) {
                swap_lists();
                set_bound(kp.max_rank, kp.n);
                tied = true;
              }
            }
            if (!tied)
              select_union(stage_keys + (size_t)b0 * VK, idx0 + b0 * VK, nb * VK, trim_slack);
          }
          SEGTOPK_STAT_ADD(kStatFirstBound, clock64() - tb);
          if (nb < nv)
            process_vectors(stage, fwd ? nb : 0u, fwd ? nv : nv - nb, idx0, release);
        }
      } else {
        process_vectors(stage, 0u, nv, idx0, release);
      }
      release();
    }
    if (threadIdx.x == 0) {
      // after a wait gave up: let every copy still in flight land before
      // this CTA's shared memory is released (each wait bounded)
      for (uint32_t s = landed; s < issued; ++s)
        mbar_wait(&ctl.bars[(gbase + s) % S], ((gbase + s) / S) & 1u, p.wait_limit);
    }
    gstep = gbase + nchunks;
    SEGTOPK_STAT_ADD(kStatChunks, nchunks);

    if (has_tail && fwd)
      offer_edge(n - tail, tail);
    if (has_head && !fwd)
      offer_edge(0, head);
    SEGTOPK_STAT_ADD(kStatStream, clock64() - t_pass);
    __syncthreads(); // the stop flag is final for this pass
    return spec_used;
  };

  const bool spec_pass = stream_pass(true);
  bool aborted = ctl.abort != 0;
  if (!aborted && spec_pass && count < min(k, n_slice)) {
    // the sample misled the bound (an ordered slice): read the slice again
    // with bounds from exact selections only
    SEGTOPK_STAT_ADD(kStatRestreams, 1);
    count = 0;
    open = true;
    bound = Bound<Raw, Rank>{(Rank)0, (Raw)0};
    __syncthreads();
    stream_pass(false);
    aborted = ctl.abort != 0;
  }
  SEGTOPK_STAT_ADD(kStatSpec, spec_pass ? 1 : 0);
  SEGTOPK_STAT_ADD(kStatKeys, n_slice);
  SEGTOPK_STAT_ADD(kStatListEntries, count);
  if (aborted && C == 1)
    return; // a wait gave up: no output (bit 0 of the device error word is set)
#ifdef SEGTOPK_STATS
  const long long t_final = clock64();
  // flushes this CTA's counters once, at every exit below
  auto flush_stats = [&]() {
    SEGTOPK_STAT_ADD(kStatFinal, clock64() - t_final);
    SEGTOPK_STAT_ADD(kStatCycles, clock64() - t_start);
    SEGTOPK_STAT_ADD(kStatDigitPasses, sel_pass);
    if (threadIdx.x == 0)
      for (int i = 0; i < kStatCount; ++i)
        if (ctl.stat[i])
          atomicAdd(&g_stats[i], ctl.stat[i]);
  };
#define SEGTOPK_FLUSH_STATS() flush_stats()
#else
#define SEGTOPK_FLUSH_STATS()                                                                      \
  do {                                                                                             \
  } while (0)
#endif

  // local top-k of this CTA's slice, for clusters that gather top-k lists
  // (a lone CTA selects once when writing the output; the histogram merge
  // works on whole lists: each holds its slice's top-k and, at the boundary
  // rank, a preference-order prefix of the slice's ties)
  __syncthreads();
  if (count > k && C > 1 && p.merge_gather == 1 && !aborted)
    trim_list(0u);

  Raw* out_keys = reinterpret_cast<Raw*>(p.out_keys) + seg * (int64_t)k;
  const int64_t vbytes = p.value_bytes;
  const ValueSink vals{p.out_values ? static_cast<char*>(p.out_values) + seg * (int64_t)k * vbytes : nullptr,
                       p.values ? static_cast<const char*>(p.values) + g0 * vbytes : nullptr, vbytes == 8 ? 1 : 0};

  // The k best of n list entries (any order), written to this segment's
  // output slots: small sets by counting, larger ones by a radix selection
  // and then a sort of the k survivors when the output is sorted.
  auto finish = [&](Raw* raw, uint32_t* idx, uint32_t nn, Raw* sp_raw, uint32_t* sp_idx, unsigned char* scratch) {
    if (nn <= kCountFinalMax) {
      finalize_small<TR, NT, kCountFinalMax>(raw, idx, nn, k, dirmask, pl, p.sorted != 0, scratch, out_keys, vals);
      return;
    }
#ifdef SEGTOPK_STATS
    const long long t_sel = clock64();
#endif
    uint32_t mm = nn; // every entry is selected when nn <= k
    if (nn > k) {
      sel_pass =
        trim_into<TR, NT>(ctl, sel_pass, list_src(raw, idx, nn), sp_raw, sp_idx, k, 0u, dirmask, pl, cbuf, tie_any).pass;
      raw = sp_raw;
      idx = sp_idx;
      mm = k;
    }
#ifdef SEGTOPK_STATS
    const long long t_write = clock64();
    SEGTOPK_STAT_ADD(kStatFinalSelect, t_write - t_sel);
    struct WriteTimer {
      Ctrl& ctl;
      long long t;
      __device__ ~WriteTimer() { SEGTOPK_STAT_ADD(kStatFinalWrite, clock64() - t); }
    } write_timer{ctl, t_write};
#endif
    if (!p.sorted) {
      for (uint32_t e = threadIdx.x; e < mm; e += NT) {
        out_keys[e] = raw[e];
        if (vals)
          vals.put(e, idx[e]);
      }
    } else if (mm <= kCountMax) {
      finalize_small<TR, NT>(raw, idx, mm, mm, dirmask, pl, true, scratch, out_keys, vals);
    } else {
      sort_and_write<TR, NT>(raw, idx, mm, dirmask, scratch, out_keys, vals, p.stable != 0);
    }
  };

  if (C == 1) {
    finish(list_raw, list_idx, count, spare_raw, spare_idx, ring);
    SEGTOPK_FLUSH_STATS();
    return;
  }

  // ---------------- cluster merge ----------------
  const uint32_t leader = 0;
  // A CTA holding its slice's exact top-k knows that the segment's k-th best
  // is no worse than its own k-th best; the best of these bounds over the
  // cluster limits what every CTA sends to the leader (worth its cost when
  // the gathered lists would be too long to finish by counting).
  const bool prune = p.merge_gather == 1 && C * k > kCountMax;
  if (prune) {
    uint64_t wr = ~0ull, wp = ~0ull; // no bound
    if (count >= k)
      list_worst<TR, NT>(ctl, list_raw, list_idx, count, dirmask, pl, wr, wp);
    if (threadIdx.x == 0) {
      const uint32_t xa = dsmem_map(smem_addr(&ctl.xb[rank][0]), leader);
      dsmem_st(xa, wr);
      dsmem_st(xa + 8u, wp);
    }
  }
  cluster_sync(); // every CTA has finished streaming and published its bound; every initialisation is visible
  {
    // a CTA whose copy wait gave up stops the whole cluster: every CTA reads
    // every CTA's flag, and all leave after one more cluster barrier
    uint32_t any = 0;
    if (threadIdx.x < C)
      any = dsmem_ld_u32(dsmem_map(smem_addr(&ctl.abort), threadIdx.x));
    if (__syncthreads_or(any != 0)) {
      cluster_sync();
      return;
    }
  }

  if (p.merge_gather) {
    if (threadIdx.x < 32) {
      uint64_t br = ~0ull, bp = ~0ull; // no bound
      if (prune && threadIdx.x < C) {
        const uint32_t xa = dsmem_map(smem_addr(&ctl.xb[threadIdx.x][0]), leader);
        br = dsmem_ld_u64(xa);
        bp = dsmem_ld_u64(xa + 8u);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t orr = __shfl_xor_sync(kFull, br, o);
        const uint64_t opp = __shfl_xor_sync(kFull, bp, o);
        if (orr < br || (orr == br && opp < bp)) {
          br = orr;
          bp = opp;
        }
      }
      if (threadIdx.x == 0) {
        ctl.xb_min[0] = br;
        ctl.xb_min[1] = bp;
      }
    }
    __syncthreads();
    const uint64_t tb_r = ctl.xb_min[0], tb_p = ctl.xb_min[1];
    // every CTA's surviving entries into the leader's ring, one warp-wide atomic per 32 entries
    const uint32_t cap = C * (p.merge_gather == 2 ? L : k);
    Raw* g_raw = reinterpret_cast<Raw*>(ring);
    uint32_t* g_idx = reinterpret_cast<uint32_t*>(ring + align16(cap * sizeof(Raw)));
    const uint32_t graw = dsmem_map(smem_addr(g_raw), leader);
    const uint32_t gidx = dsmem_map(smem_addr(g_idx), leader);
    const uint32_t gcnt = dsmem_map(smem_addr(&ctl.gather_count), leader);
    for (uint32_t base = 0; base < count; base += NT) {
      const uint32_t e = base + threadIdx.x;
      bool valid = e < count;
      if (valid) {
        const uint64_t r = (uint64_t)TR::rank(list_raw[e], dirmask);
        const uint64_t pi = pref_index(list_idx[e], pl);
        valid = r < tb_r || (r == tb_r && pi <= tb_p);
      }
      const uint32_t bal = __ballot_sync(kFull, valid);
      if (bal) {
        uint32_t wb = 0;
        if (lane_id() == 0)
          wb = dsmem_atom_add(gcnt, __popc(bal));
        wb = __shfl_sync(kFull, wb, 0);
        if (valid) {
          const uint32_t pos = wb + __popc(bal & lanemask_lt());
          dsmem_st(graw + pos * (uint32_t)sizeof(Raw), list_raw[e]);
          dsmem_st(gidx + pos * 4u, list_idx[e]);
        }
      }
    }
    cluster_sync(); // the leader holds every candidate
    if (rank != leader) {
      SEGTOPK_FLUSH_STATS();
      return;
    }
    unsigned char* scratch = ring + align16(cap * sizeof(Raw)) + align16(cap * 4u);
    finish(g_raw, g_idx, ctl.gather_count, list_raw, list_idx, scratch); // the leader's own lists are free now
    SEGTOPK_FLUSH_STATS();
    return;
  }

  // histogram merge: radix passes over the union of the lists
  Selection<Rank> sel{(Rank)0, (Rank)0, 0u, 0u};
  uint32_t ties_needed = n; // n <= k: every entry of every CTA is taken, as a boundary entry
  if (n > k) {
    constexpr int RB = TR::kRankBits;
    constexpr int P = RB / kDigitBits;
    uint32_t krem = k;
    const uint32_t merged_addr = dsmem_map(smem_addr(&ctl.hist_merged[0]), leader);
    for (int pass = 0; pass < P; ++pass) {
      const int shift = RB - kDigitBits * (pass + 1);
      for (uint32_t e = threadIdx.x; e < count; e += NT) {
        const Rank r = TR::rank(list_raw[e], dirmask);
        if ((r & sel.mask) == sel.prefix)
          atomicAdd(&ctl.hist_m0[(uint32_t)(r >> shift) & (kBuckets - 1)], 1u);
      }
      __syncthreads();
      if (rank != leader) {
        for (uint32_t i = threadIdx.x; i < (uint32_t)kBuckets; i += NT) {
          const uint32_t v = ctl.hist_m0[i];
          if (v)
            dsmem_red_add(merged_addr + 4u * i, v);
          ctl.hist_m0[i] = 0;
        }
      }
      cluster_sync(); // every fold has landed in the leader
      if (rank == leader && threadIdx.x < 32) {
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t b = 8 * threadIdx.x + i;
          h[i] = ctl.hist_merged[b] + ctl.hist_m0[b];
          ctl.hist_merged[b] = 0;
          ctl.hist_m0[b] = 0;
        }
        find_bucket(h, krem, ctl.res);
      }
      cluster_sync(); // the pass result is published
      uint32_t b, before, cnt;
      if (rank == leader) {
        b = ctl.res[0];
        before = ctl.res[1];
        cnt = ctl.res[2];
      } else {
        const uint32_t ra = dsmem_map(smem_addr(&ctl.res[0]), leader);
        b = dsmem_ld_u32(ra);
        before = dsmem_ld_u32(ra + 4);
        cnt = dsmem_ld_u32(ra + 8);
      }
      krem -= before;
      sel.prefix |= (Rank)b << shift;
      sel.mask |= (Rank)(kBuckets - 1) << shift;
      if (cnt == krem)
        break;
    }
    ties_needed = krem;
  }
  const uint32_t f_total = m - ties_needed;

  // cross-CTA count scan in preference order
  const Src<Raw> lsrc = list_src(list_raw, list_idx, count);
  const uint2 tot = scan_list<TR, NT>(
    ctl, lsrc, dirmask,
    [&](uint32_t, Raw, uint32_t, Rank rk) {
      const Rank mr = rk & sel.mask;
      return mr < sel.prefix ? 1 : (mr == sel.prefix ? 2 : 0);
    },
    [](uint32_t, Raw, uint32_t, Rank, int, uint32_t, uint32_t) {});
  const uint32_t my_pos = fwd ? rank : C - 1 - rank;
  if (threadIdx.x < C) {
    const uint32_t d = threadIdx.x;
    const uint32_t d_pos = fwd ? d : C - 1 - d;
    if (d_pos > my_pos) {
      if (tot.x)
        dsmem_red_add(dsmem_map(smem_addr(&ctl.front_base), d), tot.x);
      if (tot.y)
        dsmem_red_add(dsmem_map(smem_addr(&ctl.tie_base), d), tot.y);
    }
  }
  cluster_sync(); // every CTA's bases are final
  const uint32_t fbase = ctl.front_base, tbase = ctl.tie_base;

  // this CTA's share of the boundary ties, chosen by source index (any of
  // them in the not_guaranteed mode: the first `quota` in list order)
  const uint32_t quota = ties_needed > tbase ? min(tot.y, ties_needed - tbase) : 0u;
  if (quota > 0 && quota < tot.y && !tie_any)
  {
    CandBuf cb = cbuf;
    cb.n = ~0u;
    select_ties<TR, NT>(ctl, sel_pass, lsrc, quota, dirmask, pl, sel, cb);
  }
  const bool take_ties = quota > 0;
  auto classify = [&](uint32_t, Raw, uint32_t ki, Rank rk) {
    const int c = sel.classify(rk, pref_index(ki, pl));
    return (c == 2 && !take_ties) ? 0 : c;
  };
  auto position = [&](int cls, uint32_t r1, uint32_t r2) {
    return cls == 1 ? fbase + r1 : f_total + tbase + r2;
  };

  if (!p.sorted) {
    scan_list<TR, NT>(ctl, lsrc, dirmask, classify,
                      [&](uint32_t, Raw kr, uint32_t ki, Rank, int cls, uint32_t r1, uint32_t r2) {
                        if (cls == 2 && r2 >= quota)
                          return; // a surplus tie (not_guaranteed)
                        const uint32_t pos = position(cls, r1, r2);
                        out_keys[pos] = kr;
                        if (vals)
                          vals.put(pos, ki);
                      });
    SEGTOPK_FLUSH_STATS();
    return;
  }

  // sorted: gather the m selected items into the leader's ring, the leader sorts
  Raw* g_raw = reinterpret_cast<Raw*>(ring);
  uint32_t* g_idx = reinterpret_cast<uint32_t*>(ring + align16(m * sizeof(Raw)));
  unsigned char* scratch = ring + align16(m * sizeof(Raw)) + align16(m * 4u);
  const uint32_t graw = dsmem_map(smem_addr(g_raw), leader);
  const uint32_t gidx = dsmem_map(smem_addr(g_idx), leader);
  scan_list<TR, NT>(ctl, lsrc, dirmask, classify,
                    [&](uint32_t, Raw kr, uint32_t ki, Rank, int cls, uint32_t r1, uint32_t r2) {
                      if (cls == 2 && r2 >= quota)
                        return; // a surplus tie (not_guaranteed)
                      const uint32_t pos = position(cls, r1, r2);
                      dsmem_st(graw + pos * (uint32_t)sizeof(Raw), kr);
                      dsmem_st(gidx + pos * 4u, ki);
                    });
  cluster_sync(); // the leader holds all m items
  if (rank != leader) {
    SEGTOPK_FLUSH_STATS();
    return;
  }
  sort_and_write<TR, NT>(g_raw, g_idx, m, dirmask, scratch, out_keys, vals, p.stable != 0);
  SEGTOPK_FLUSH_STATS();
#undef SEGTOPK_FLUSH_STATS
}

} // namespace segtopk
