// Shared device helpers for the segmented top-k kernels (sm_103a).
//
// Inline PTX for: 1-D bulk copies (TMA) driven by mbarriers, thread-block
// cluster barriers and distributed shared memory (DSMEM) access, plus the
// order-preserving key transform and its raw-domain superset filter.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace segtopk {

// ---------------------------------------------------------------------------
// Device error word (read and cleared by segtopk_read_device_error).
// ---------------------------------------------------------------------------
enum : uint32_t {
  kErrCopyTimeout = 1u,   // an mbarrier wait on a bulk copy gave up
  kErrSegmentTooLong = 2u // a segment exceeded the planned length class
};
// One error word per translation unit (read by that unit's host accessor).
static __device__ uint32_t g_device_error;

__device__ __forceinline__ void raise_error(uint32_t bits) { atomicOr(&g_device_error, bits); }

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy (TMA, 1-D). dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
  asm volatile(
    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
      smem_addr(dst)),
    "l"(src), "r"(bytes), "r"(smem_addr(bar))
    : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
  uint32_t ok;
  asm volatile(
    "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
    : "=r"(ok)
    : "r"(smem_addr(bar)), "r"(parity)
    : "memory");
  return ok != 0;
}

// As mbar_try_wait, with the thread suspended for at most about `ns`
// nanoseconds while the phase is incomplete (so that a polling loop around
// it also notices other events soon).
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns)
{
  uint32_t ok;
  asm volatile(
    "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
    : "=r"(ok)
    : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
    : "memory");
  return ok != 0;
}

// Default bound of a wait on a bulk copy: about one second of SM clock cycles.
constexpr long long kWaitLimitCycles = 1ll << 31;

// Bounded wait on the phase of `bar` with the given parity: gives up after
// `limit` SM clock cycles and records the failure in the device error word.
// Callers make the outcome uniform (one waiting lane, broadcast) before
// branching on it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kWaitLimitCycles)
{
  if (mbar_try_wait(bar, parity))
    return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > limit) {
      raise_error(kErrCopyTimeout);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// Thread-block clusters and DSMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x()
{
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive()
{
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync()
{
  cluster_arrive();
  cluster_wait();
}
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_smem_addr, uint32_t rank)
{
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_red_add(uint32_t addr, uint32_t v)
{
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v)
{
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr)
{
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t dsmem_ld_u64(uint32_t addr)
{
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint16_t v)
{
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v)
{
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint64_t v)
{
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Order-preserving key transform.
//
// T maps a key's bits to an unsigned integer whose order is the key's numeric
// order: floats flip the sign bit of non-negative values and invert all bits
// of negative ones; -0.0 is first replaced by +0.0 so that both zeros get one
// code ("Fix BlockTopK +/-0.0 handling", Cause: canonicalise the zero before
// any direction handling, never compare raw bits against extracted digits).
// Signed integers flip the sign bit; unsigned integers are unchanged.
//
// The selection works on the rank code r = T(x) XOR dirmask, where dirmask is
// all ones for "max" and zero for "min", so that a smaller r is always a
// better key. XOR-ing every bit reverses every radix digit, i.e. the bucket
// index b becomes num_buckets-1-b for the max direction -- the bucket
// reversal of the same page's Fix section -- and the raw key bits are only
// ever copied, never compared as ranks.
//
// Each key kind provides
//   rank(x, dirmask)       the rank code (smaller = better);
//   unrank(r, dirmask)     raw bits of a key with rank r (never -0.0);
//   pass_bits(v, braw, brank, is_max)
//                          per key of a 16-byte vector, a bit that is set
//                          for every key ranking below brank (and may be set
//                          for NaNs and, for 64-bit keys, keys whose high
//                          word ties braw's); key_of_bit(q) is the key
//                          behind bit q;
//   may_pass(v, braw, brank, is_max, strict)
//                          for a 16-byte vector of keys: false only if no key
//                          in it ranks below brank (strict) or at most brank
//                          (not strict), where braw are the bits of a key
//                          whose rank is brank. It may answer true for keys
//                          that then fail the exact test (ties, NaNs), never
//                          false for one that passes. Floats use one native
//                          compare per key against braw ("better than" or
//                          "not worse than", both also true for NaN);
//                          integers the exact test on the rank.
// ---------------------------------------------------------------------------
// A rank bound in both domains: a key enters iff its rank is below tau;
// raw holds the bits of a key whose rank is tau (the raw-domain filter).
template <class Raw, class Rank>
struct Bound {
  Rank tau;
  Raw raw;
};

enum class KeyKind : int { F16 = 0, BF16 = 1, F32 = 2, F64 = 3, U32 = 4, I32 = 5 };

template <KeyKind K>
struct KeyTraits;

// IEEE floats of 16, 32 or 64 bits.
template <class Raw, int BITS>
struct FloatRank {
  static constexpr Raw kSign = (Raw)((Raw)1 << (BITS - 1));
  __device__ __forceinline__ static Raw t(Raw x)
  {
    const Raw v = (x == kSign) ? (Raw)0 : x; // -0.0 -> +0.0
    const Raw neg = (Raw)((Raw)0 - (Raw)(v >> (BITS - 1)));
    return (Raw)(v ^ (Raw)(neg | kSign));
  }
  __device__ __forceinline__ static Raw t_inv(Raw t)
  {
    return (t & kSign) ? (Raw)(t & (Raw)~kSign) : (Raw)~t;
  }
};

// Eight 16-bit lanes' compare masks (0xffff per true half) to one bit per
// key: bits 0-3 are the low halves of words 0-3 (keys 0, 2, 4, 6), bits 4-7
// the high halves (keys 1, 3, 5, 7).
__device__ __forceinline__ uint32_t half_mask_bits(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3)
{
  const uint32_t b = (m0 & 0x00010001u) | ((m1 & 0x00010001u) << 1) | ((m2 & 0x00010001u) << 2) |
                     ((m3 & 0x00010001u) << 3);
  return (b & 0xfu) | (b >> 12);
}
__device__ __forceinline__ uint32_t half_key_of_bit(uint32_t q) { return q < 4u ? 2u * q : 2u * (q - 4u) + 1u; }

template <>
struct KeyTraits<KeyKind::F16> {
  using Raw = uint16_t;
  using Rank = uint32_t;
  static constexpr int kRankBits = 16;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask)
  {
    return ((Rank)FloatRank<uint16_t, 16>::t(x)) ^ dirmask;
  }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask)
  {
    return FloatRank<uint16_t, 16>::t_inv((uint16_t)(r ^ dirmask));
  }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw braw, Rank, bool is_max)
  {
    const __half e = __ushort_as_half(braw);
    const __half2 h = __halves2half2(e, e);
    const __half2* w = reinterpret_cast<const __half2*>(&v);
    if (is_max)
      return half_mask_bits(__hgtu2_mask(w[0], h), __hgtu2_mask(w[1], h), __hgtu2_mask(w[2], h), __hgtu2_mask(w[3], h));
    return half_mask_bits(__hltu2_mask(w[0], h), __hltu2_mask(w[1], h), __hltu2_mask(w[2], h), __hltu2_mask(w[3], h));
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return half_key_of_bit(q); }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw braw, Rank, bool is_max, bool strict)
  {
    const __half e = __ushort_as_half(braw);
    const __half2 h = __halves2half2(e, e);
    const __half2* w = reinterpret_cast<const __half2*>(&v);
    unsigned m;
    if (is_max)
      m = strict ? (__hgtu2_mask(w[0], h) | __hgtu2_mask(w[1], h) | __hgtu2_mask(w[2], h) | __hgtu2_mask(w[3], h))
                 : (__hgeu2_mask(w[0], h) | __hgeu2_mask(w[1], h) | __hgeu2_mask(w[2], h) | __hgeu2_mask(w[3], h));
    else
      m = strict ? (__hltu2_mask(w[0], h) | __hltu2_mask(w[1], h) | __hltu2_mask(w[2], h) | __hltu2_mask(w[3], h))
                 : (__hleu2_mask(w[0], h) | __hleu2_mask(w[1], h) | __hleu2_mask(w[2], h) | __hleu2_mask(w[3], h));
    return m != 0;
  }
};

template <>
struct KeyTraits<KeyKind::BF16> {
  using Raw = uint16_t;
  using Rank = uint32_t;
  static constexpr int kRankBits = 16;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask)
  {
    return ((Rank)FloatRank<uint16_t, 16>::t(x)) ^ dirmask;
  }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask)
  {
    return FloatRank<uint16_t, 16>::t_inv((uint16_t)(r ^ dirmask));
  }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw braw, Rank, bool is_max)
  {
    const __nv_bfloat16 e = __ushort_as_bfloat16(braw);
    const __nv_bfloat162 h = __halves2bfloat162(e, e);
    const __nv_bfloat162* w = reinterpret_cast<const __nv_bfloat162*>(&v);
    if (is_max)
      return half_mask_bits(__hgtu2_mask(w[0], h), __hgtu2_mask(w[1], h), __hgtu2_mask(w[2], h), __hgtu2_mask(w[3], h));
    return half_mask_bits(__hltu2_mask(w[0], h), __hltu2_mask(w[1], h), __hltu2_mask(w[2], h), __hltu2_mask(w[3], h));
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return half_key_of_bit(q); }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw braw, Rank, bool is_max, bool strict)
  {
    const __nv_bfloat16 e = __ushort_as_bfloat16(braw);
    const __nv_bfloat162 h = __halves2bfloat162(e, e);
    const __nv_bfloat162* w = reinterpret_cast<const __nv_bfloat162*>(&v);
    unsigned m;
    if (is_max)
      m = strict ? (__hgtu2_mask(w[0], h) | __hgtu2_mask(w[1], h) | __hgtu2_mask(w[2], h) | __hgtu2_mask(w[3], h))
                 : (__hgeu2_mask(w[0], h) | __hgeu2_mask(w[1], h) | __hgeu2_mask(w[2], h) | __hgeu2_mask(w[3], h));
    else
      m = strict ? (__hltu2_mask(w[0], h) | __hltu2_mask(w[1], h) | __hltu2_mask(w[2], h) | __hltu2_mask(w[3], h))
                 : (__hleu2_mask(w[0], h) | __hleu2_mask(w[1], h) | __hleu2_mask(w[2], h) | __hleu2_mask(w[3], h));
    return m != 0;
  }
};

template <>
struct KeyTraits<KeyKind::F32> {
  using Raw = uint32_t;
  using Rank = uint32_t;
  static constexpr int kRankBits = 32;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask) { return FloatRank<uint32_t, 32>::t(x) ^ dirmask; }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask)
  {
    return FloatRank<uint32_t, 32>::t_inv(r ^ dirmask);
  }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw braw, Rank, bool is_max)
  {
    const float f = __uint_as_float(braw);
    const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
    const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
    if (is_max)
      return (uint32_t)!(x0 <= f) | ((uint32_t)!(x1 <= f) << 1) | ((uint32_t)!(x2 <= f) << 2) |
             ((uint32_t)!(x3 <= f) << 3);
    return (uint32_t)!(x0 >= f) | ((uint32_t)!(x1 >= f) << 1) | ((uint32_t)!(x2 >= f) << 2) |
           ((uint32_t)!(x3 >= f) << 3);
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return q; }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw braw, Rank, bool is_max, bool strict)
  {
    const float f = __uint_as_float(braw);
    const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
    const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
    if (is_max) {
      if (strict)
        return !(x0 <= f) | !(x1 <= f) | !(x2 <= f) | !(x3 <= f);
      return !(x0 < f) | !(x1 < f) | !(x2 < f) | !(x3 < f);
    }
    if (strict)
      return !(x0 >= f) | !(x1 >= f) | !(x2 >= f) | !(x3 >= f);
    return !(x0 > f) | !(x1 > f) | !(x2 > f) | !(x3 > f);
  }
};

template <>
struct KeyTraits<KeyKind::F64> {
  using Raw = uint64_t;
  using Rank = uint64_t;
  static constexpr int kRankBits = 64;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask) { return FloatRank<uint64_t, 64>::t(x) ^ dirmask; }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask)
  {
    return FloatRank<uint64_t, 64>::t_inv(r ^ dirmask);
  }
  // The high word of a double as a signed integer in the double's own order
  // (sign-magnitude to two's complement); -0.0 lands one below +0.0, which
  // only widens the superset test below.
  __device__ __forceinline__ static int32_t order_hi(uint32_t hi)
  {
    const int32_t x = (int32_t)hi;
    return x ^ (int32_t)((uint32_t)(x >> 31) >> 1);
  }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw braw, Rank, bool is_max)
  {
    const uint32_t bh = (uint32_t)(braw >> 32);
    // the usual cases in the raw high words: a bound at or above +0.0 for
    // max (a better key is positive, and positive doubles order like their
    // bits as signed integers), a negative bound for min (a better key is
    // negative, and larger magnitudes have larger unsigned bits)
    if (is_max && (int32_t)bh >= 0)
      return (uint32_t)((int32_t)v.y >= (int32_t)bh) | ((uint32_t)((int32_t)v.w >= (int32_t)bh) << 1);
    if (!is_max && (int32_t)bh < 0)
      return (uint32_t)(v.y >= bh) | ((uint32_t)(v.w >= bh) << 1);
    const int32_t ob = order_hi(bh);
    const int32_t o0 = order_hi(v.y), o1 = order_hi(v.w);
    if (is_max)
      return (uint32_t)(o0 >= ob) | ((uint32_t)(o1 >= ob) << 1);
    return (uint32_t)(o0 <= ob) | ((uint32_t)(o1 <= ob) << 1);
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return q; }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw braw, Rank, bool is_max, bool)
  {
    // a key ranking at most the bound is, as a number, at least (max) or at
    // most (min) the bound key, so its high word compares likewise (one
    // compare of the high words cannot be strict, so this test never is)
    const int32_t ob = order_hi((uint32_t)(braw >> 32));
    const int32_t o0 = order_hi(v.y), o1 = order_hi(v.w);
    if (is_max)
      return (o0 >= ob) | (o1 >= ob);
    return (o0 <= ob) | (o1 <= ob);
  }
};

template <>
struct KeyTraits<KeyKind::U32> {
  using Raw = uint32_t;
  using Rank = uint32_t;
  static constexpr int kRankBits = 32;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask) { return x ^ dirmask; }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask) { return r ^ dirmask; }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw, Rank brank, bool is_max)
  {
    const uint32_t dm = is_max ? 0xffffffffu : 0u; // exact
    return (uint32_t)((v.x ^ dm) < brank) | ((uint32_t)((v.y ^ dm) < brank) << 1) |
           ((uint32_t)((v.z ^ dm) < brank) << 2) | ((uint32_t)((v.w ^ dm) < brank) << 3);
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return q; }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw, Rank brank, bool is_max, bool strict)
  {
    const uint32_t dm = is_max ? 0xffffffffu : 0u; // exact
    if (strict)
      return ((v.x ^ dm) < brank) | ((v.y ^ dm) < brank) | ((v.z ^ dm) < brank) | ((v.w ^ dm) < brank);
    return ((v.x ^ dm) <= brank) | ((v.y ^ dm) <= brank) | ((v.z ^ dm) <= brank) | ((v.w ^ dm) <= brank);
  }
};

template <>
struct KeyTraits<KeyKind::I32> {
  using Raw = uint32_t;
  using Rank = uint32_t;
  static constexpr int kRankBits = 32;
  __device__ __forceinline__ static Rank rank(Raw x, Rank dirmask) { return (x ^ 0x80000000u) ^ dirmask; }
  __device__ __forceinline__ static Raw unrank(Rank r, Rank dirmask) { return (r ^ dirmask) ^ 0x80000000u; }
  __device__ __forceinline__ static uint32_t pass_bits(const uint4& v, Raw, Rank brank, bool is_max)
  {
    const uint32_t dm = (is_max ? 0xffffffffu : 0u) ^ 0x80000000u; // exact
    return (uint32_t)((v.x ^ dm) < brank) | ((uint32_t)((v.y ^ dm) < brank) << 1) |
           ((uint32_t)((v.z ^ dm) < brank) << 2) | ((uint32_t)((v.w ^ dm) < brank) << 3);
  }
  __device__ __forceinline__ static uint32_t key_of_bit(uint32_t q) { return q; }
  __device__ __forceinline__ static bool may_pass(const uint4& v, Raw, Rank brank, bool is_max, bool strict)
  {
    const uint32_t dm = (is_max ? 0xffffffffu : 0u) ^ 0x80000000u; // exact
    if (strict)
      return ((v.x ^ dm) < brank) | ((v.y ^ dm) < brank) | ((v.z ^ dm) < brank) | ((v.w ^ dm) < brank);
    return ((v.x ^ dm) <= brank) | ((v.y ^ dm) <= brank) | ((v.z ^ dm) <= brank) | ((v.w ^ dm) <= brank);
  }
};

// ---------------------------------------------------------------------------
// Keys of a 16-byte vector held in registers
// ---------------------------------------------------------------------------
// Key j of a 16-byte vector, and the vector with key j set (j is a
// compile-time constant after unrolling; no local-memory views of registers).
template <class Raw>
__device__ __forceinline__ uint32_t vec_word(const uint4& v, int w)
{
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}
template <class Raw>
__device__ __forceinline__ Raw vec_key(const uint4& v, int j)
{
  if constexpr (sizeof(Raw) == 8)
    return ((uint64_t)vec_word<Raw>(v, 2 * j + 1) << 32) | vec_word<Raw>(v, 2 * j);
  else if constexpr (sizeof(Raw) == 4)
    return vec_word<Raw>(v, j);
  else
    return (Raw)(vec_word<Raw>(v, j >> 1) >> (16 * (j & 1)));
}
__device__ __forceinline__ void vec_or_word(uint4& v, int w, uint32_t x)
{
  if (w == 0)
    v.x |= x;
  else if (w == 1)
    v.y |= x;
  else if (w == 2)
    v.z |= x;
  else
    v.w |= x;
}
template <class Raw>
__device__ __forceinline__ void vec_set_key(uint4& v, int j, Raw x) // slot j holds zero
{
  if constexpr (sizeof(Raw) == 8) {
    vec_or_word(v, 2 * j, (uint32_t)x);
    vec_or_word(v, 2 * j + 1, (uint32_t)((uint64_t)x >> 32));
  } else if constexpr (sizeof(Raw) == 4) {
    vec_or_word(v, j, (uint32_t)x);
  } else {
    vec_or_word(v, j >> 1, (uint32_t)x << (16 * (j & 1)));
  }
}

// Where a segment's selected values go: out[pos] receives the payload of
// the element at segment-local index idx -- in[idx] with 4- or 8-byte
// values, or, with no payload array (an internal mode of the host-buffer
// entry point), idx itself. A sink with no output (keys only) is false.
struct ValueSink {
  void* out;      // this segment's output values (null: keys only)
  const void* in; // this segment's input values (null: write source indices)
  int wide;       // 8-byte values
  __device__ __forceinline__ explicit operator bool() const { return out != nullptr; }
  __device__ __forceinline__ void put(uint32_t pos, uint32_t idx) const
  {
    if (wide)
      static_cast<int64_t*>(out)[pos] = in ? static_cast<const int64_t*>(in)[idx] : (int64_t)idx;
    else
      static_cast<int32_t*>(out)[pos] = in ? static_cast<const int32_t*>(in)[idx] : (int32_t)idx;
  }
};

// ---------------------------------------------------------------------------
// Warp helpers
// ---------------------------------------------------------------------------
constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t lanemask_lt()
{
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t x)
{
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= (uint32_t)o)
      x += y;
  }
  return x;
}

template <typename T>
__device__ __forceinline__ T warp_max(T x)
{
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    T y = __shfl_xor_sync(kFull, x, o);
    x = y > x ? y : x;
  }
  return x;
}

} // namespace segtopk
