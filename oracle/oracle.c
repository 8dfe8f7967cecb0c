/*
 * CPU oracle for segmented (batched) top-k.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of the result, written out:
 *
 *   For each segment s = [offsets[s], offsets[s+1]) (empty when end <= begin,
 *   per "Implement Segmented TopK using Thread-Block-Clusters", bot walkthrough
 *   "Bug Fixes": negative segment sizes are treated as empty) with local
 *   indices i = 0..n-1:
 *
 *   1. Keys are compared as numbers. +0.0 and -0.0 compare equal ("Fix
 *      BlockTopK +/-0.0 handling", Cause and Fix: both zeros must land in the
 *      same bucket), but each element keeps its own bit pattern in the output.
 *   2. Selection order: better key first (larger for max, smaller for min);
 *      among equal keys the preferred source index first -- smaller index for
 *      prefer_smaller_index, larger index for prefer_larger_index ("Top-K:
 *      Determinism, Tie-Breaking, and Output Ordering", "Tie-break" table).
 *      An unspecified tie-break is read as prefer_smaller_index (that page's
 *      "Which items are selected?" leaves the choice to the implementation).
 *   3. The first m = min(k, n) elements of that order are selected.
 *   4. Output order (same page, "Output ordering" table): stable_sorted sorts
 *      the selected items by key, better first, equal keys by source index
 *      ascending (input order) whatever the tie-break; "sorted" is written the
 *      same way (a valid refinement); "unsorted" is also written in that
 *      order here and compared as a set by the tests.
 *   5. out_keys[s*k + j] holds the original bits of the j-th output element,
 *      out_values[s*k + j] = values[offsets[s] + index]; slots j >= m are left
 *      untouched.
 *
 * NaN keys (the pages are silent): a NaN with the sign bit clear ranks above
 * +inf, one with the sign bit set below -inf; two positive NaNs order by
 * their payload ascending, two negative NaNs by payload descending.
 *
 * The sort is a plain top-down merge sort written here; its comparator is a
 * total order (indices are distinct), so the result does not depend on the
 * sort's stability.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Key type codes understood by this oracle. */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_F64 = 3, ORC_U32 = 4, ORC_I32 = 5 };
enum { ORC_MAX = 0, ORC_MIN = 1 };
enum { ORC_TIE_UNSPECIFIED = 0, ORC_TIE_SMALLER = 1, ORC_TIE_LARGER = 2 };

/* ---------- decoding keys to comparable numbers ---------- */

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint32_t h)
{
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32. */
double oracle_decode_bf16(uint32_t h)
{
  uint32_t w = (h & 0xffffu) << 16;
  float x;
  memcpy(&x, &w, 4);
  return (double)x;
}

typedef struct {
  int nan_class;    /* -1: NaN with sign set, 0: not NaN, +1: NaN with sign clear */
  uint64_t payload; /* NaN fraction bits (used only to order NaNs of one sign) */
  double num;       /* numeric value for floating types */
  int64_t inum;     /* exact value for integer types */
} key_val;

static key_val decode_key(int dtype, const void* keys, int64_t pos)
{
  key_val r;
  r.nan_class = 0;
  r.payload = 0;
  r.num = 0.0;
  r.inum = 0;
  switch (dtype) {
  case ORC_F16: {
    uint16_t h = ((const uint16_t*)keys)[pos];
    r.num = oracle_decode_f16(h);
    if (isnan(r.num)) {
      r.nan_class = (h & 0x8000u) ? -1 : 1;
      r.payload = h & 0x3ffu;
    }
    break;
  }
  case ORC_BF16: {
    uint16_t h = ((const uint16_t*)keys)[pos];
    r.num = oracle_decode_bf16(h);
    if (isnan(r.num)) {
      r.nan_class = (h & 0x8000u) ? -1 : 1;
      r.payload = h & 0x7fu;
    }
    break;
  }
  case ORC_F32: {
    uint32_t w = ((const uint32_t*)keys)[pos];
    float x;
    memcpy(&x, &w, 4);
    r.num = (double)x;
    if (isnan(x)) {
      r.nan_class = (w & 0x80000000u) ? -1 : 1;
      r.payload = w & 0x7fffffu;
    }
    break;
  }
  case ORC_F64: {
    uint64_t w = ((const uint64_t*)keys)[pos];
    double x;
    memcpy(&x, &w, 8);
    r.num = x;
    if (isnan(x)) {
      r.nan_class = (w >> 63) ? -1 : 1;
      r.payload = w & 0xfffffffffffffull;
    }
    break;
  }
  case ORC_U32:
    r.inum = (int64_t)((const uint32_t*)keys)[pos];
    break;
  case ORC_I32:
  default:
    r.inum = (int64_t)((const int32_t*)keys)[pos];
    break;
  }
  return r;
}

/* Numeric three-way comparison in ascending order: -1 if a < b, 0 if equal, +1 if a > b. */
static int compare_ascending(int dtype, const key_val* a, const key_val* b)
{
  if (dtype == ORC_U32 || dtype == ORC_I32)
    return (a->inum > b->inum) - (a->inum < b->inum);
  if (a->nan_class != 0 || b->nan_class != 0) {
    if (a->nan_class != b->nan_class)
      return (a->nan_class > b->nan_class) ? 1 : -1;
    /* same sign of NaN */
    if (a->payload == b->payload)
      return 0;
    if (a->nan_class > 0)
      return (a->payload > b->payload) ? 1 : -1;
    return (a->payload > b->payload) ? -1 : 1;
  }
  /* +0.0 == -0.0 under C's numeric comparison */
  return (a->num > b->num) - (a->num < b->num);
}

/* ---------- merge sort of local indices under a total order ---------- */

typedef struct {
  int dtype;
  int direction;
  int tie;            /* ORC_TIE_* for selection, ignored in output order */
  int output_order;   /* 1: equal keys by index ascending; 0: by tie preference */
  const key_val* vals;
} order_ctx;

/* Returns nonzero iff local index a comes strictly before local index b. */
static int comes_first(const order_ctx* c, int64_t a, int64_t b)
{
  int ab = compare_ascending(c->dtype, &c->vals[a], &c->vals[b]);
  if (ab != 0)
    return (c->direction == ORC_MAX) ? (ab > 0) : (ab < 0);
  if (c->output_order || c->tie != ORC_TIE_LARGER)
    return a < b;
  return a > b;
}

static void merge_sort(const order_ctx* c, int64_t* a, int64_t* tmp, int64_t n)
{
  if (n < 2)
    return;
  int64_t h = n / 2;
  merge_sort(c, a, tmp, h);
  merge_sort(c, a + h, tmp, n - h);
  int64_t i = 0, j = h, o = 0;
  while (i < h && j < n) {
    if (comes_first(c, a[j], a[i]))
      tmp[o++] = a[j++];
    else
      tmp[o++] = a[i++];
  }
  while (i < h)
    tmp[o++] = a[i++];
  while (j < n)
    tmp[o++] = a[j++];
  memcpy(a, tmp, (size_t)n * sizeof(int64_t));
}

static size_t key_size(int dtype)
{
  switch (dtype) {
  case ORC_F16:
  case ORC_BF16:
    return 2;
  case ORC_F64:
    return 8;
  default:
    return 4;
  }
}

/*
 * Top-k of segments [seg_lo, seg_hi). Returns 0 on success, -1 on bad
 * arguments, -2 when memory could not be obtained.
 */
int oracle_batched_topk(int dtype, const void* keys, const int32_t* values, const int64_t* offsets,
                        int64_t seg_lo, int64_t seg_hi, int32_t k, int direction, int tie_break,
                        void* out_keys, int32_t* out_values)
{
  if (dtype < ORC_F16 || dtype > ORC_I32 || k < 0 || seg_lo < 0 || seg_hi < seg_lo)
    return -1;
  if (direction != ORC_MAX && direction != ORC_MIN)
    return -1;
  if (tie_break < ORC_TIE_UNSPECIFIED || tie_break > ORC_TIE_LARGER)
    return -1;
  const size_t ks = key_size(dtype);
  for (int64_t s = seg_lo; s < seg_hi; ++s) {
    const int64_t begin = offsets[s];
    const int64_t end = offsets[s + 1];
    const int64_t n = end > begin ? end - begin : 0;
    const int64_t m = n < (int64_t)k ? n : (int64_t)k;
    if (m == 0)
      continue;
    key_val* vals = (key_val*)malloc((size_t)n * sizeof(key_val));
    int64_t* idx = (int64_t*)malloc((size_t)n * sizeof(int64_t));
    int64_t* tmp = (int64_t*)malloc((size_t)n * sizeof(int64_t));
    if (!vals || !idx || !tmp) {
      free(vals);
      free(idx);
      free(tmp);
      return -2;
    }
    for (int64_t i = 0; i < n; ++i) {
      vals[i] = decode_key(dtype, keys, begin + i);
      idx[i] = i;
    }
    order_ctx c;
    c.dtype = dtype;
    c.direction = direction;
    c.tie = tie_break;
    c.vals = vals;
    /* selection: the first m under (better key, preferred index) */
    c.output_order = 0;
    merge_sort(&c, idx, tmp, n);
    /* output: the selected m under (better key, index ascending) */
    c.output_order = 1;
    merge_sort(&c, idx, tmp, m);
    for (int64_t j = 0; j < m; ++j) {
      const int64_t src = begin + idx[j];
      memcpy((char*)out_keys + ((size_t)s * (size_t)k + (size_t)j) * ks,
             (const char*)keys + (size_t)src * ks, ks);
      if (values && out_values)
        out_values[s * (int64_t)k + j] = values[src];
    }
    free(vals);
    free(idx);
    free(tmp);
  }
  return 0;
}
