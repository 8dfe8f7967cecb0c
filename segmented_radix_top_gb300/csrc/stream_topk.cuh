// The segment kernel: one CTA, or one thread-block cluster, per segment.
//
// Method ("Implement Segmented TopK using Thread-Block-Clusters", sections
// 1.2 - 1.6 and 2): multi-pass radix digit selection with a final filter that
// writes the keys strictly beyond the splitter plus exactly enough boundary
// ties, ties taken in source-index order.
//
// GB300 design (what differs from the pages' CUB kernel):
//  * Keys stream once from HBM through a ring of 16 KiB shared-memory stages
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

constexpr uint32_t kChunkBytes = 16384;

struct KernelParams {
  const void* keys;
  const int32_t* values;
  const int64_t* offsets;
  void* out_keys;
  int32_t* out_values;
  int64_t num_segments;
  int64_t n_lo;          // this launch serves segments with n_lo < n <= n_hi
  int64_t n_hi;
  uint64_t dirmask;      // rank = T(key) ^ dirmask: all ones for max, zero for min
  int32_t k;
  uint32_t list_cap;     // candidate list capacity (entries)
  uint32_t trim_at;      // trim when the list holds more than this after a chunk
  uint32_t ring_stages;  // pipeline depth (<= 8)
  uint32_t ring_bytes;   // ring region bytes (also sort / gather scratch)
  int32_t prefer_larger; // tie preference: larger source index first
  int32_t sorted;        // write the selected items in stable sorted order
  int32_t merge_gather;  // cluster merge by gathering every CTA's list into the leader
  int32_t flag_overlong; // report segments longer than n_hi
};

// Host and device agree on the dynamic shared-memory layout.
__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }
__host__ __device__ inline uint32_t list_bytes(uint32_t cap, uint32_t key_bytes)
{
  return align16(cap * key_bytes) + cap * 4u;
}

template <KeyKind KK, int NT>
__global__ void __launch_bounds__(NT, 2) stream_topk_kernel(const KernelParams p)
{
  using TR = KeyTraits<KK>;
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  constexpr int VK = 16 / (int)sizeof(Raw);     // keys per 16-byte vector
  constexpr int U = (int)kChunkBytes / 16 / NT; // vectors per thread per chunk
  constexpr uint32_t kChunkVec = kChunkBytes / 16;
  static_assert(U >= 1 && U <= 8, "chunk / thread configuration");

  extern __shared__ __align__(128) unsigned char smem[];
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem);
  unsigned char* ring = smem + kCtrlBytes;
  Raw* list_raw = reinterpret_cast<Raw*>(ring + p.ring_bytes);
  uint32_t* list_idx = reinterpret_cast<uint32_t*>(ring + p.ring_bytes + align16(p.list_cap * sizeof(Raw)));

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
  const uint32_t n = (uint32_t)n64;
  const uint32_t k = (uint32_t)p.k;
  const uint32_t m = k < n ? k : n;
  const Rank dirmask = (Rank)p.dirmask;
  const bool is_max = dirmask != 0;
  const bool fwd = !p.prefer_larger;
  const uint32_t S = p.ring_stages;

  // ---- front-loaded shared-memory initialisation ----
  for (uint32_t i = threadIdx.x; i < kBuckets; i += NT) {
    ctl.hist[0][i] = 0;
    ctl.hist[1][i] = 0;
    ctl.hist_merged[i] = 0;
  }
  if (threadIdx.x == 0) {
    ctl.list_count = 0;
    ctl.gather_count = 0;
    ctl.front_base = 0;
    ctl.tie_base = 0;
    for (uint32_t s = 0; s < S; ++s)
      mbar_init(&ctl.bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this CTA's slice of the segment ----
  const Raw* seg_keys = reinterpret_cast<const Raw*>(p.keys) + g0;
  uint32_t head = (uint32_t)((VK - (int)(g0 % VK)) % VK); // unaligned leading keys
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

  auto chunk_of_step = [&](uint32_t s) { return fwd ? s : nchunks - 1 - s; };
  auto issue = [&](uint32_t s) {
    const uint32_t v0 = v_lo + chunk_of_step(s) * kChunkVec;
    const uint32_t nv = min(kChunkVec, v_hi - v0);
    const uint32_t st = s % S;
    mbar_arrive_expect_tx(&ctl.bars[st], nv * 16u);
    bulk_load(ring + (size_t)st * kChunkBytes, seg_keys + head + (size_t)v0 * VK, nv * 16u, &ctl.bars[st]);
  };
  uint32_t issued = 0;
  if (threadIdx.x == 0) {
    for (; issued < S && issued < nchunks; ++issued)
      issue(issued);
  }

  // ---- streaming selection state (uniform across the block) ----
  bool open = true; // no bound yet: every key is accepted
  Bound<Raw, Rank> bound{(Rank)0, (Raw)0};

  // Offer this thread's U vectors (vector j: vc[j] keys from slot 0, source
  // indices i0[j] + slot) to the list. Returns true in every lane of a warp
  // whose appends pushed the list past the trim threshold.
  auto offer = [&](const uint4 (&vec)[U], const uint32_t (&vc)[U], const uint32_t (&i0)[U]) {
    bool may = false;
#pragma unroll
    for (int j = 0; j < U; ++j)
      if (vc[j])
        may = may || open || TR::may_pass(vec[j], bound, is_max);
    bool over = false;
    if (__any_sync(kFull, may)) {
      uint32_t acc[U];
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        acc[j] = 0;
        if (may) {
          const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
          for (int i = 0; i < VK; ++i)
            if ((uint32_t)i < vc[j] && (open || TR::rank(kv[i], dirmask) < bound.tau))
              acc[j] |= 1u << i;
        }
        c += __popc(acc[j]);
      }
      const uint32_t incl = warp_inclusive_sum(c);
      const uint32_t tot = __shfl_sync(kFull, incl, 31);
      if (tot) {
        uint32_t base = 0;
        if (lane_id() == 31)
          base = atomicAdd(&ctl.list_count, tot);
        base = __shfl_sync(kFull, base, 31);
        uint32_t pos = base + incl - c;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
          for (int i = 0; i < VK; ++i) {
            if ((acc[j] >> i) & 1u) {
              list_raw[pos] = kv[i];
              list_idx[pos] = i0[j] + (uint32_t)i;
              ++pos;
            }
          }
        }
        over = base + tot > p.trim_at;
      }
    }
    return over;
  };

  // After a chunk: trim when the next chunk could overflow the list.
  auto after_chunk = [&](bool over) {
    const uint32_t count = ctl.list_count;
    (void)over;
    const Rank tau = trim_list<TR, NT>(ctl, list_raw, list_idx, count, k, dirmask, p.prefer_larger != 0);
    bound.tau = tau;
    bound.raw = TR::unrank(tau, dirmask);
    open = false;
  };

  // Unaligned head / tail keys: plain loads, one per thread.
  auto offer_edge = [&](uint32_t e_begin, uint32_t e_cnt) {
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
    if (__syncthreads_or(offer(vec, vc, i0)))
      after_chunk(true);
  };

  if (has_head && fwd)
    offer_edge(0, head);
  if (has_tail && !fwd)
    offer_edge(n - tail, tail);

  bool copies_ok = true;
  for (uint32_t s = 0; s < nchunks; ++s) {
    const uint32_t st = s % S;
    if (copies_ok)
      copies_ok = mbar_wait(&ctl.bars[st], (s / S) & 1u);
    const uint32_t vb = v_lo + chunk_of_step(s) * kChunkVec;
    const uint32_t nv = min(kChunkVec, v_hi - vb);
    const uint4* stage = reinterpret_cast<const uint4*>(ring + (size_t)st * kChunkBytes);
    uint4 vec[U];
    uint32_t vc[U], i0[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t t = (uint32_t)j * NT + threadIdx.x;
      const bool ok = t < nv && copies_ok;
      vec[j] = ok ? stage[t] : make_uint4(0, 0, 0, 0);
      vc[j] = ok ? (uint32_t)VK : 0u;
      i0[j] = head + (vb + t) * VK;
    }
    const bool over = offer(vec, vc, i0);
    const int any_over = __syncthreads_or(over); // also ends every read of this stage
    if (threadIdx.x == 0 && copies_ok && issued < nchunks) {
      issue(issued); // refill the stage just released
      ++issued;
    }
    if (any_over)
      after_chunk(true);
  }
  if (!copies_ok && threadIdx.x == 0) {
    // let every copy still in flight land before this CTA's shared memory is released
    for (uint32_t s = 0; s < issued; ++s)
      mbar_wait(&ctl.bars[s % S], (s / S) & 1u);
  }

  if (has_tail && fwd)
    offer_edge(n - tail, tail);
  if (has_head && !fwd)
    offer_edge(0, head);

  // local top-k of this CTA's slice
  __syncthreads();
  uint32_t count = ctl.list_count;
  if (count > k) {
    trim_list<TR, NT>(ctl, list_raw, list_idx, count, k, dirmask, p.prefer_larger != 0);
    count = k;
  }

  Raw* out_keys = reinterpret_cast<Raw*>(p.out_keys) + seg * (int64_t)k;
  int32_t* out_values = p.out_values ? p.out_values + seg * (int64_t)k : nullptr;
  const int32_t* values = p.values ? p.values + g0 : nullptr;

  if (C == 1) {
    // count == m: the list is the answer
    if (p.sorted) {
      sort_and_write<TR, NT>(list_raw, list_idx, count, dirmask, ring, out_keys, out_values, values);
    } else {
      for (uint32_t e = threadIdx.x; e < count; e += NT) {
        out_keys[e] = list_raw[e];
        if (out_values)
          out_values[e] = values[list_idx[e]];
      }
    }
    return;
  }

  // ---------------- cluster merge ----------------
  const uint32_t leader = 0;
  cluster_sync(); // every CTA has finished streaming; every CTA's initialisation is visible

  if (p.merge_gather) {
    // every CTA's list (<= k entries) into the leader's ring, one warp-wide atomic per 32 entries
    const uint32_t cap = C * k;
    Raw* g_raw = reinterpret_cast<Raw*>(ring);
    uint32_t* g_idx = reinterpret_cast<uint32_t*>(ring + align16(cap * sizeof(Raw)));
    const uint32_t graw = dsmem_map(smem_addr(g_raw), leader);
    const uint32_t gidx = dsmem_map(smem_addr(g_idx), leader);
    const uint32_t gcnt = dsmem_map(smem_addr(&ctl.gather_count), leader);
    for (uint32_t base = 0; base < count; base += NT) {
      const uint32_t e = base + threadIdx.x;
      const bool valid = e < count;
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
    if (rank != leader)
      return;
    uint32_t total = ctl.gather_count;
    if (total > k) {
      trim_list<TR, NT>(ctl, g_raw, g_idx, total, k, dirmask, p.prefer_larger != 0);
      total = k;
    }
    unsigned char* scratch = ring + align16(cap * sizeof(Raw)) + align16(cap * 4u);
    if (p.sorted) {
      sort_and_write<TR, NT>(g_raw, g_idx, total, dirmask, scratch, out_keys, out_values, values);
    } else {
      for (uint32_t e = threadIdx.x; e < total; e += NT) {
        out_keys[e] = g_raw[e];
        if (out_values)
          out_values[e] = values[g_idx[e]];
      }
    }
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
          atomicAdd(&ctl.hist[0][(uint32_t)(r >> shift) & (kBuckets - 1)], 1u);
      }
      __syncthreads();
      if (rank != leader && threadIdx.x < kBuckets) {
        const uint32_t v = ctl.hist[0][threadIdx.x];
        if (v)
          dsmem_red_add(merged_addr + 4u * threadIdx.x, v);
        ctl.hist[0][threadIdx.x] = 0;
      }
      cluster_sync(); // every fold has landed in the leader
      if (rank == leader && threadIdx.x < 32) {
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t b = 8 * threadIdx.x + i;
          h[i] = ctl.hist_merged[b] + ctl.hist[0][b];
          ctl.hist_merged[b] = 0;
          ctl.hist[0][b] = 0;
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
  const uint2 tot = scan_list<TR, NT>(
    ctl, list_raw, list_idx, count, dirmask,
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

  // this CTA's share of the boundary ties, chosen by source index
  const uint32_t quota = ties_needed > tbase ? min(tot.y, ties_needed - tbase) : 0u;
  if (quota > 0 && quota < tot.y)
    select_ties<TR, NT>(ctl, list_raw, list_idx, count, quota, dirmask, p.prefer_larger != 0, sel);
  const bool take_ties = quota > 0;
  auto classify = [&](uint32_t, Raw, uint32_t ki, Rank rk) {
    const int c = sel.classify(rk, pref_index(ki, p.prefer_larger != 0));
    return (c == 2 && !take_ties) ? 0 : c;
  };
  auto position = [&](int cls, uint32_t r1, uint32_t r2) {
    return cls == 1 ? fbase + r1 : f_total + tbase + r2;
  };

  if (!p.sorted) {
    scan_list<TR, NT>(ctl, list_raw, list_idx, count, dirmask, classify,
                      [&](uint32_t, Raw kr, uint32_t ki, Rank, int cls, uint32_t r1, uint32_t r2) {
                        const uint32_t pos = position(cls, r1, r2);
                        out_keys[pos] = kr;
                        if (out_values)
                          out_values[pos] = values[ki];
                      });
    return;
  }

  // sorted: gather the m selected items into the leader's ring, the leader sorts
  Raw* g_raw = reinterpret_cast<Raw*>(ring);
  uint32_t* g_idx = reinterpret_cast<uint32_t*>(ring + align16(m * sizeof(Raw)));
  unsigned char* scratch = ring + align16(m * sizeof(Raw)) + align16(m * 4u);
  const uint32_t graw = dsmem_map(smem_addr(g_raw), leader);
  const uint32_t gidx = dsmem_map(smem_addr(g_idx), leader);
  scan_list<TR, NT>(ctl, list_raw, list_idx, count, dirmask, classify,
                    [&](uint32_t, Raw kr, uint32_t ki, Rank, int cls, uint32_t r1, uint32_t r2) {
                      const uint32_t pos = position(cls, r1, r2);
                      dsmem_st(graw + pos * (uint32_t)sizeof(Raw), kr);
                      dsmem_st(gidx + pos * 4u, ki);
                    });
  cluster_sync(); // the leader holds all m items
  if (rank != leader)
    return;
  sort_and_write<TR, NT>(g_raw, g_idx, m, dirmask, scratch, out_keys, out_values, values);
}

} // namespace segtopk
