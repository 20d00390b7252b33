/*
 * CPU oracle for the deterministic W-way bf16 reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * What it computes (arx.cu, `arx_kernel`, the reduce loop and its "rank order:
 * every rank gets the same bits" comment): for every element i,
 *
 *     acc = +0.0f
 *     for r = 0 .. W-1:   acc = fl32(acc + widen(slot[r][i]))
 *     out[i] = bf16_rne(acc)
 *
 * widen() is the exact bf16 -> fp32 conversion (`__bfloat162float` in the
 * page), bf16_rne() is the single rounding to bf16, round to nearest with ties
 * to even (`__float2bfloat16` in the page).  Each fp32 add is the host's IEEE
 * binary32 add in round-to-nearest-even; the build uses no fast-math and
 * oracle_fp_env_ok() checks at load time that subnormals are not flushed.
 *
 * Readings where the page is silent (each also listed in the design notes):
 *  - NaN: the page never produces one; here a NaN result is encoded as the
 *    quiet NaN 0x7FC0 with the input's sign.  Comparisons treat NaN payloads
 *    as unpinned (NaN-ness only).
 *  - Overflow: a finite fp32 sum whose rounding exceeds the largest bf16
 *    rounds to +-inf, as round-to-nearest does in IEEE 754.
 *  - W may be 1 (the page requires W >= 2); the definition is unchanged.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 *        -pthread (no target-specific flags; builds on x86-64 and aarch64).
 */
#include <fenv.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 <-> fp32 --------------------------------------------------------
 * bf16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits,
 * 7 fraction bits.  Widening appends 16 zero fraction bits, which is exact.
 */
static float widen_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a binary32 to the nearest bf16, ties to even (IEEE 754
 * roundTiesToEven applied to a 7-bit fraction).  The 16 dropped bits are
 * compared against one half ulp of the kept part (0x8000).  Adding one to the
 * kept 16-bit pattern moves to the next representable magnitude; a carry out
 * of the fraction correctly bumps the exponent, and from the largest finite
 * value it lands on infinity (0x7F80 / 0xFF80), which is what rounding to
 * nearest does past the overflow threshold. */
static uint16_t round_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  const uint32_t exponent = (u >> 23) & 0xFFu;
  const uint32_t fraction = u & 0x7FFFFFu;
  if (exponent == 0xFFu && fraction != 0u) {
    return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u); /* quiet NaN, sign kept */
  }
  uint32_t kept = u >> 16;
  const uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) {
    kept += 1u;
  }
  return (uint16_t)kept;
}

/* ---- the reduce ---------------------------------------------------------- */

/* One element range of the reduce.  i-outer, r-inner, exactly as defined
 * above.  Every slot value at i is read before out[i] is written, so `out`
 * may be one of the slots. */
static void reduce_range(const uint16_t* const* slots, int W, uint16_t* out,
                         size_t lo, size_t hi) {
  for (size_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int r = 0; r < W; ++r) {
      acc = acc + widen_bf16(slots[r][i]);
    }
    out[i] = round_bf16_rne(acc);
  }
}

typedef struct {
  const uint16_t* const* slots;
  int W;
  uint16_t* out;
  size_t lo, hi;
} range_job;

static void* range_worker(void* p) {
  const range_job* j = (const range_job*)p;
  reduce_range(j->slots, j->W, j->out, j->lo, j->hi);
  return NULL;
}

/* out[i] = bf16_rne(sum over r in rank order of widen(slots[r][i])).
 * slots: W host pointers to n uint16 bf16 patterns each.  Returns 0, or -1 on
 * invalid arguments. */
int oracle_reduce(const uint16_t* const* slots, int W, uint16_t* out, size_t n) {
  if (W < 1 || !slots || (n && !out)) return -1;
  for (int r = 0; r < W; ++r)
    if (n && !slots[r]) return -1;
  reduce_range(slots, W, out, 0, n);
  return 0;
}

/* The same definition with the element range split over `threads` POSIX
 * threads.  Each element is still summed by one thread in rank order, so the
 * result is identical to oracle_reduce(); only the wall time changes. */
int oracle_reduce_mt(const uint16_t* const* slots, int W, uint16_t* out,
                     size_t n, int threads) {
  if (threads <= 1 || n < 4096) return oracle_reduce(slots, W, out, n);
  if (W < 1 || !slots || !out) return -1;
  for (int r = 0; r < W; ++r)
    if (!slots[r]) return -1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  range_job jobs[256];
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    jobs[t].slots = slots;
    jobs[t].W = W;
    jobs[t].out = out;
    jobs[t].lo = n / (size_t)threads * (size_t)t;
    jobs[t].hi = t == threads - 1 ? n : n / (size_t)threads * (size_t)(t + 1);
    if (pthread_create(&tid[t], NULL, range_worker, &jobs[t]) != 0) {
      reduce_range(slots, W, out, jobs[t].lo, jobs[t].hi); /* run inline */
      tid[t] = 0;
      continue;
    }
    ++started;
  }
  for (int t = 0; t < threads; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
  (void)started;
  return 0;
}

/* Reduce over a [W][n] row-major block of patterns (slot r starts at
 * base + r*n).  Convenience for callers holding one contiguous array. */
int oracle_reduce_rows(const uint16_t* base, int W, uint16_t* out, size_t n,
                       int threads) {
  if (W < 1 || W > 64) return -1;
  const uint16_t* slots[64];
  for (int r = 0; r < W; ++r) slots[r] = base + (size_t)r * n;
  return oracle_reduce_mt(slots, W, out, n, threads);
}

/* ---- conversions exposed for the pins -------------------------------------- */

void oracle_round_bf16_array(const float* in, uint16_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = round_bf16_rne(in[i]);
}

/* Round every binary32 bit pattern in [first, first + count) and write the
 * bf16 patterns; used to check the rounding over all 2^32 inputs in chunks. */
void oracle_round_bf16_patterns(uint32_t first, uint16_t* out, size_t count) {
  for (size_t i = 0; i < count; ++i) {
    uint32_t u = first + (uint32_t)i;
    float f;
    memcpy(&f, &u, sizeof f);
    out[i] = round_bf16_rne(f);
  }
}

void oracle_widen_bf16_array(const uint16_t* in, float* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = widen_bf16(in[i]);
}

/* fp32 sum of two binary32 values in the host's arithmetic, exposed so that
 * the tests can confirm the host add is IEEE round-to-nearest-even. */
float oracle_add_f32(float a, float b) { return a + b; }

/* ---- floating-point environment check -----------------------------------------
 * Returns 1 when the host rounds to nearest and keeps subnormals: the sum of
 * the two smallest positive subnormals must be exactly twice the smallest.  A
 * flush-to-zero or denormals-are-zero mode fails this. */
int oracle_fp_env_ok(void) {
  if (fegetround() != FE_TONEAREST) return 0;
  volatile uint32_t one_ulp = 1u;
  volatile float tiny;
  uint32_t u = one_ulp;
  float t;
  memcpy(&t, &u, sizeof t);
  tiny = t;
  volatile float sum = tiny + tiny;
  float s = sum;
  uint32_t su;
  memcpy(&su, &s, sizeof su);
  return su == 2u;
}
