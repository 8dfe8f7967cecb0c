// The segment kernel: one CTA, or one thread-block cluster, per segment.
//
// Method ("Implement Segmented TopK using Thread-Block-Clusters", sections
// 1.2 - 1.6 and 2): multi-pass radix digit selection with a final filter that
// writes the keys strictly beyond the splitter plus exactly enough boundary
// ties, ties taken in source-index order.
//
// GB300 design (what differs from the pages' CUB kernel):
//  * Keys are streamed once from HBM through a ring of 16 KiB shared-memory
//    stages filled by 1-D bulk copies (TMA) with one mbarrier per stage.
//  * Instead of keeping the whole segment resident and re-reading it every
//    pass, each CTA keeps a bounded candidate list in shared memory that
//    always contains the best k keys of what it has read so far, in
//    preference order. A key enters the list only if it beats the current
//    bound (the rank of the k-th best key kept); when the list is about to
//    overflow it is trimmed back to k entries by the same radix digit
//    selection, which also tightens the bound. Every key is read from HBM
//    exactly once and, after the first few chunks, costs one compare.
//  * A cluster of C CTAs splits a long segment into C contiguous slices; the
//    slices' candidate lists are merged by the pages' cluster mechanism:
//    per-CTA digit histograms folded into the leader CTA through DSMEM, the
//    leader's scan broadcast back, a cross-CTA count scan of (front, tie)
//    counts in preference order, and, for sorted output, a DSMEM gather of
//    the selected items into the leader, which sorts and writes them.
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
  uint32_t ring_stages;  // pipeline depth (<= 8)
  uint32_t ring_bytes;   // ring region bytes (also sort / gather scratch)
  int32_t prefer_larger; // tie preference: larger source index first
  int32_t sorted;        // write the selected items in stable sorted order
  int32_t flag_overlong; // report segments longer than n_hi
};

// Host and device agree on the dynamic shared-memory layout.
template <int KB>
__host__ __device__ inline uint32_t list_raw_bytes(uint32_t cap)
{
  return (cap * KB + 15u) & ~15u;
}
template <int KB>
__host__ __device__ inline uint32_t smem_bytes(uint32_t ring_bytes, uint32_t cap)
{
  return kCtrlBytes + ring_bytes + list_raw_bytes<KB>(cap) + cap * 4u;
}

template <KeyKind KK, int NT>
__global__ void __launch_bounds__(NT, 2) stream_topk_kernel(const KernelParams p)
{
  using TR = KeyTraits<KK>;
  using Raw = typename TR::Raw;
  using Rank = typename TR::Rank;
  constexpr int VK = 16 / (int)sizeof(Raw);           // keys per 16-byte vector
  constexpr int U = (int)kChunkBytes / 16 / NT;       // vectors per thread per chunk
  constexpr uint32_t kChunkVec = kChunkBytes / 16;
  constexpr int NW = NT / 32;
  static_assert(U >= 1 && U <= 4, "chunk / thread configuration");

  extern __shared__ __align__(128) unsigned char smem[];
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem);
  unsigned char* ring = smem + kCtrlBytes;
  Raw* list_raw = reinterpret_cast<Raw*>(ring + p.ring_bytes);
  uint32_t* list_idx = reinterpret_cast<uint32_t*>(ring + p.ring_bytes + list_raw_bytes<sizeof(Raw)>(p.list_cap));

  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int64_t seg = (C == 1) ? (int64_t)blockIdx.x : (int64_t)cluster_id_x();
  if (seg >= p.num_segments)
    return;
  const int64_t g0 = p.offsets[seg];
  const int64_t g1 = p.offsets[seg + 1];
  const int64_t n64 = g1 > g0 ? g1 - g0 : 0;
  if (n64 <= p.n_lo)
    return; // another launch serves this segment (whole cluster returns)
  if (n64 > p.n_hi) {
    if (p.flag_overlong && threadIdx.x == 0 && rank == 0)
      raise_error(kErrSegmentTooLong);
    return;
  }
  const uint32_t n = (uint32_t)n64;
  const uint32_t k = (uint32_t)p.k;
  const uint32_t m = k < n ? k : n;
  const Rank dirmask = (Rank)p.dirmask;
  const bool fwd = !p.prefer_larger;
  const uint32_t S = p.ring_stages;

  // ---- front-loaded shared-memory initialisation ----
  for (uint32_t i = threadIdx.x; i < kBuckets; i += NT) {
    ctl.hist[0][i] = 0;
    ctl.hist[1][i] = 0;
    ctl.hist_merged[i] = 0;
  }
  if (threadIdx.x == 0) {
    ctl.front_base = 0;
    ctl.tie_base = 0;
    for (uint32_t s = 0; s < S; ++s)
      mbar_init(&ctl.bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (C > 1)
    cluster_arrive(); // publishes the zeroed counters; the matching wait precedes the first DSMEM access

  // ---- this CTA's slice of the segment ----
  const Raw* seg_keys = reinterpret_cast<const Raw*>(p.keys) + g0;
  uint32_t head = (uint32_t)((VK - (int)(g0 % VK)) % VK);
  if (head > n)
    head = n;
  const uint32_t body_v = (n - head) / VK;
  const uint32_t tail = n - head - body_v * VK;
  const uint32_t v_lo = (uint32_t)(((uint64_t)body_v * rank) / C);
  const uint32_t v_hi = (uint32_t)(((uint64_t)body_v * (rank + 1)) / C);
  const uint32_t nvec = v_hi - v_lo;
  const uint32_t nchunks = (nvec + kChunkVec - 1) / kChunkVec;
  const bool has_head = rank == 0 && head > 0;
  const bool has_tail = rank == C - 1 && tail > 0;

  // chunk processed at step s (processing order = preference order)
  auto chunk_of_step = [&](uint32_t s) { return fwd ? s : nchunks - 1 - s; };
  auto issue = [&](uint32_t s) {
    const uint32_t ci = chunk_of_step(s);
    const uint32_t v0 = v_lo + ci * kChunkVec;
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

  bool copies_ok = true;
  // ---- streaming selection state (uniform across the block) ----
  uint32_t count = 0;  // list entries
  bool open = true;    // no bound yet: accept everything
  Rank tau = 0;        // accept a key iff open || rank < tau
  int sbuf = 0;        // scan_tot buffer
  const uint32_t L = p.list_cap;

  // Offer this thread's keys (U vectors; vector j holds vc[j] valid keys in
  // processing order starting at slot fwd ? 0 : VK-1 with source index
  // i0[j] stepping +1 / -1) to the candidate list. The block-wide barrier at
  // its start ends all reads of the ring stage of step `issue_step` (< 0 for
  // the edge elements), whose stage is then refilled with step + S.
  auto ingest = [&](const uint4 (&vec)[U], const uint32_t (&vc)[U], const uint32_t (&i0)[U],
                    int issue_step) {
    uint32_t acc[U];
    uint64_t packed = 0;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      acc[j] = 0;
      const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
      for (int i = 0; i < VK; ++i) {
        const int slot = fwd ? i : VK - 1 - i;
        const Rank r = TR::rank(kv[slot], dirmask);
        if ((uint32_t)i < vc[j] && (open || r < tau))
          acc[j] |= 1u << i;
      }
      packed |= (uint64_t)__popc(acc[j]) << (16 * j);
    }
    const int any = __syncthreads_or(packed != 0);
    if (issue_step >= 0 && threadIdx.x == 0 && copies_ok && issued < nchunks &&
        issued == (uint32_t)issue_step + S) {
      issue(issued); // the stage just read is free again
      ++issued;
    }
    if (!any)
      return;
    for (;;) {
      // ordered positions: block exclusive scan of the packed per-round counts
      const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
      uint64_t incl = packed;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= (uint32_t)o)
          incl += y;
      }
      if (lane == 31)
        ctl.scan_tot[sbuf][warp] = incl;
      __syncthreads();
      uint64_t excl = incl - packed, total = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const uint64_t v = ctl.scan_tot[sbuf][w];
        if (w < (int)warp)
          excl += v;
        total += v;
      }
      sbuf ^= 1;
      uint32_t tot_all = 0;
#pragma unroll
      for (int j = 0; j < U; ++j)
        tot_all += (uint32_t)(total >> (16 * j)) & 0xffffu;
      if (count + tot_all > L) {
        // make room: trim the list to its k best and tighten the bound
        tau = trim_list<TR, NT>(ctl, list_raw, list_idx, count, k, dirmask);
        count = k;
        open = false;
        packed = 0;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
          uint32_t a = 0;
#pragma unroll
          for (int i = 0; i < VK; ++i) {
            const int slot = fwd ? i : VK - 1 - i;
            if (((acc[j] >> i) & 1u) && TR::rank(kv[slot], dirmask) < tau)
              a |= 1u << i;
          }
          acc[j] = a;
          packed |= (uint64_t)__popc(a) << (16 * j);
        }
        continue;
      }
      uint32_t round_base = count;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        uint32_t pos = round_base + ((uint32_t)(excl >> (16 * j)) & 0xffffu);
        const Raw* kv = reinterpret_cast<const Raw*>(&vec[j]);
#pragma unroll
        for (int i = 0; i < VK; ++i) {
          if ((acc[j] >> i) & 1u) {
            const int slot = fwd ? i : VK - 1 - i;
            list_raw[pos] = kv[slot];
            list_idx[pos] = fwd ? i0[j] + i : i0[j] - i;
            ++pos;
          }
        }
        round_base += (uint32_t)(total >> (16 * j)) & 0xffffu;
      }
      count += tot_all;
      return;
    }
  };

  // Unaligned head / tail elements: loaded with plain loads, one per thread.
  auto ingest_edge = [&](uint32_t e_begin, uint32_t e_cnt) {
    uint4 vec[U];
    uint32_t vc[U], i0[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      vec[j] = make_uint4(0, 0, 0, 0);
      vc[j] = 0;
      i0[j] = 0;
    }
    if (threadIdx.x < e_cnt) {
      const uint32_t e = fwd ? e_begin + threadIdx.x : e_begin + e_cnt - 1 - threadIdx.x;
      Raw* kv = reinterpret_cast<Raw*>(&vec[0]);
      kv[fwd ? 0 : VK - 1] = seg_keys[e];
      vc[0] = 1;
      i0[0] = e;
    }
    ingest(vec, vc, i0, -1);
  };

  if (has_head && fwd)
    ingest_edge(0, head);
  if (has_tail && !fwd)
    ingest_edge(n - tail, tail);

  for (uint32_t s = 0; s < nchunks; ++s) {
    const uint32_t st = s % S;
    if (copies_ok)
      copies_ok = mbar_wait(&ctl.bars[st], (s / S) & 1u);
    const uint32_t ci = chunk_of_step(s);
    const uint32_t vb = v_lo + ci * kChunkVec;
    const uint32_t nv = min(kChunkVec, v_hi - vb);
    const uint4* stage = reinterpret_cast<const uint4*>(ring + (size_t)st * kChunkBytes);
    uint4 vec[U];
    uint32_t vc[U], i0[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t t = (uint32_t)j * NT + threadIdx.x;
      if (t < nv && copies_ok) {
        const uint32_t cv = fwd ? t : nv - 1 - t;
        vec[j] = stage[cv];
        vc[j] = VK;
        i0[j] = head + (vb + cv) * VK + (fwd ? 0u : (uint32_t)(VK - 1));
      } else {
        vec[j] = make_uint4(0, 0, 0, 0);
        vc[j] = 0;
        i0[j] = 0;
      }
    }
    ingest(vec, vc, i0, (int)s);
  }
  if (!copies_ok && threadIdx.x == 0) {
    // let every copy still in flight land before this CTA's shared memory is released
    for (uint32_t s = 0; s < issued; ++s)
      mbar_wait(&ctl.bars[s % S], (s / S) & 1u);
  }

  if (has_tail && fwd)
    ingest_edge(n - tail, tail);
  if (has_head && !fwd)
    ingest_edge(0, head);

  // local top-k of this CTA's slice
  if (count > k) {
    trim_list<TR, NT>(ctl, list_raw, list_idx, count, k, dirmask);
    count = k;
  }

  Raw* out_keys = reinterpret_cast<Raw*>(p.out_keys) + seg * (int64_t)k;
  int32_t* out_values = p.out_values ? p.out_values + seg * (int64_t)k : nullptr;
  const int32_t* values = p.values ? p.values + g0 : nullptr;

  if (C == 1) {
    // count == m: the list is the answer, in preference order
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

  // ---- cluster merge ----
  cluster_wait(); // peers' initialisation is visible from here on
  const uint32_t leader = 0;
  Rank prefix = 0, mask = 0;
  uint32_t ties = n; // n <= k: every entry of every CTA is taken, as a "tie"
  if (n > k) {
    constexpr int RB = TR::kRankBits;
    constexpr int P = RB / kDigitBits;
    uint32_t krem = k;
    const uint32_t merged_addr = dsmem_map(smem_addr(&ctl.hist_merged[0]), leader);
    for (int pass = 0; pass < P; ++pass) {
      const int shift = RB - kDigitBits * (pass + 1);
      build_hist<TR, NT>(list_raw, count, dirmask, prefix, mask, shift, ctl.hist[0]);
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
      prefix |= (Rank)b << shift;
      mask |= (Rank)(kBuckets - 1) << shift;
      if (cnt == krem)
        break;
    }
    ties = krem;
  }
  const uint32_t f_total = m - ties;

  // cross-CTA count scan in preference order
  const uint2 tot = scan_list<TR, NT>(ctl, list_raw, list_idx, count, dirmask, prefix, mask,
                                      [](uint32_t, Raw, uint32_t, Rank, bool, uint32_t, uint32_t) {});
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

  if (!p.sorted) {
    scan_list<TR, NT>(ctl, list_raw, list_idx, count, dirmask, prefix, mask,
                      [&](uint32_t, Raw kr, uint32_t ki, Rank, bool isf, uint32_t fr, uint32_t tr) {
                        uint32_t pos;
                        if (isf) {
                          pos = fbase + fr;
                        } else {
                          const uint32_t g = tbase + tr;
                          if (g >= ties)
                            return;
                          pos = f_total + g;
                        }
                        out_keys[pos] = kr;
                        if (out_values)
                          out_values[pos] = values[ki];
                      });
    return;
  }

  // sorted: gather the m selected items into the leader's ring, leader sorts
  Raw* g_raw = reinterpret_cast<Raw*>(ring);
  uint32_t* g_idx = reinterpret_cast<uint32_t*>(ring + ((m * sizeof(Raw) + 15u) & ~15u));
  unsigned char* scratch = ring + ((m * sizeof(Raw) + 15u) & ~15u) + ((m * 4u + 15u) & ~15u);
  const uint32_t graw_addr = dsmem_map(smem_addr(g_raw), leader);
  const uint32_t gidx_addr = dsmem_map(smem_addr(g_idx), leader);
  scan_list<TR, NT>(ctl, list_raw, list_idx, count, dirmask, prefix, mask,
                    [&](uint32_t, Raw kr, uint32_t ki, Rank, bool isf, uint32_t fr, uint32_t tr) {
                      uint32_t pos;
                      if (isf) {
                        pos = fbase + fr;
                      } else {
                        const uint32_t g = tbase + tr;
                        if (g >= ties)
                          return;
                        pos = f_total + g;
                      }
                      dsmem_st(graw_addr + pos * (uint32_t)sizeof(Raw), kr);
                      dsmem_st(gidx_addr + pos * 4u, ki);
                    });
  cluster_sync(); // the leader holds all m items
  if (rank != leader)
    return;
  sort_and_write<TR, NT>(g_raw, g_idx, m, dirmask, scratch, out_keys, out_values, values);
}

} // namespace segtopk
