/*
 * Oracle for the virtual-rank bf16 allreduce.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, single-threaded CPU definition of what the
 * GPU library computes.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it; the library itself never does,
 * and this file shares no code, header or table with the CUDA sources.
 *
 * What is computed.  Allreduce leaves in every rank's output the element-wise
 * sum of all ranks' input buffers; the pages show it this way:
 *   - "optimize allreduce write mode by broadcast output ptr" (ROCm/aiter
 *     #1910), Motivation: stage 2 writes the reduced data into every rank's
 *     output through their output pointers;
 *   - "One shot all reduce Example" (pytorch-labs/helion #245), performance
 *     table: one-shot allreduce reads every peer's buffer and reduces locally;
 *   - "Add monolithic fused packet allreduce kernel and
 *     Model::all_reduce_packet API" (microsoft/ark #254), Changes: scatter,
 *     reduce, broadcast fused into one kernel.
 * None of the pages fixes the arithmetic.  The reading used everywhere here:
 *   acc = float(in_0[i]); acc = acc + float(in_r[i]) for r = 1 .. R-1 in rank
 *   order (plain fp32 adds, no fused multiply-add, no reassociation);
 *   out_r[i] = round-to-nearest-even bf16 of acc, the same for every r.
 * The accumulator is seeded with rank 0's value rather than +0.0 so that
 * R = 1 is the identity on every bit pattern (including -0.0).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math
 *        -fexcess-precision=standard -fPIC -shared oracle.c -o liboracle.so
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* bf16 -> fp32 is exact: a bf16 value is the upper half of an fp32 word. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * fp32 -> bf16, IEEE 754 round to nearest, ties to even.
 *
 * For a finite x, the two bf16 values that bracket |x| are `lower`, the
 * encoding whose magnitude is the largest bf16 magnitude <= |x| (the upper 16
 * bits of x), and `lower + 1`, the next larger magnitude (which is infinity
 * when `lower` is the largest finite bf16).  Within one binade, and across
 * the subnormal/normal boundary, both grids are uniform and the 16 dropped
 * bits are the distance from `lower` to |x| in units of 2^-16 of a bf16
 * spacing, so 0x8000 is exactly the midpoint.  Nearer wins; a tie goes to
 * the candidate with an even (zero) last significand bit.  The sign bit is
 * carried through unchanged.
 *
 * NaN has no nearest value; it becomes a quiet NaN with the sign and the top
 * payload bits kept.  +-inf maps to +-inf (dropped bits are zero).
 */
uint16_t oracle_f32_to_bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  const uint32_t exponent = (u >> 23) & 0xFFu;
  const uint32_t significand = u & 0x7FFFFFu;
  if (exponent == 0xFFu && significand != 0u) {
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  const uint32_t lower = u >> 16;
  const uint32_t dropped = u & 0xFFFFu;
  const uint32_t midpoint = 0x8000u;
  uint32_t result;
  if (dropped < midpoint) {
    result = lower;
  } else if (dropped > midpoint) {
    result = lower + 1u;
  } else {
    result = (lower & 1u) ? lower + 1u : lower;
  }
  return (uint16_t)result;
}

float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

/* Element-wise conversion of an array; used by the exhaustive rounding pin. */
void oracle_f32_to_bf16_array(const float* x, uint16_t* y, size_t n) {
  for (size_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16_rne(x[i]);
}

/*
 * The allreduce itself.  in[r] and out[r] are R host buffers of `count` bf16
 * words.  For each element the inputs are read before any output at that
 * element is written, so out[r] == in[r] (in place) is allowed.  Returns 0,
 * or -1 on an argument outside R in [1, 64].
 */
int oracle_allreduce_bf16(int R, size_t count, const uint16_t* const* in,
                          uint16_t* const* out) {
  if (R < 1 || R > 64) return -1;
  for (size_t i = 0; i < count; ++i) {
    float acc = bf16_to_f32(in[0][i]);
    for (int r = 1; r < R; ++r) {
      acc = acc + bf16_to_f32(in[r][i]);
    }
    const uint16_t y = oracle_f32_to_bf16_rne(acc);
    for (int r = 0; r < R; ++r) out[r][i] = y;
  }
  return 0;
}

/*
 * Reduce-scatter: the same summation, but rank r keeps only block r.  Rank
 * s's input holds R blocks of `recvcount` elements; rank r's output holds
 *   out[r][j] = bf16_rne(sum over s in rank order of in[s][r*recvcount + j]).
 * This is the one-shot push-reduce kernel of "Add HIP-graph capture coverage
 * for the sharded-relay collectives" (meta-pytorch/torchcomms #3850, the
 * commit that generalises the one-shot kernel to allreduce) with a per-peer
 * source stride of one block and an owner offset of the rank's slot times one
 * block; its allreduce case, a stride of zero, is the function above.  Outputs
 * must not overlap inputs.
 */
int oracle_reduce_scatter_bf16(int R, size_t recvcount, const uint16_t* const* in,
                               uint16_t* const* out) {
  if (R < 1 || R > 64) return -1;
  for (int r = 0; r < R; ++r) {
    const size_t base = (size_t)r * recvcount;
    for (size_t j = 0; j < recvcount; ++j) {
      float acc = bf16_to_f32(in[0][base + j]);
      for (int s = 1; s < R; ++s) acc = acc + bf16_to_f32(in[s][base + j]);
      out[r][j] = oracle_f32_to_bf16_rne(acc);
    }
  }
  return 0;
}

/*
 * All-gather: every rank's output is the concatenation, in rank order, of
 * all ranks' inputs of `sendcount` elements: out[r][s*sendcount + j] =
 * in[s][j].  No arithmetic.  Outputs must not overlap inputs.
 */
int oracle_all_gather_bf16(int R, size_t sendcount, const uint16_t* const* in,
                           uint16_t* const* out) {
  if (R < 1 || R > 64) return -1;
  for (int r = 0; r < R; ++r)
    for (int s = 0; s < R; ++s)
      for (size_t j = 0; j < sendcount; ++j) out[r][(size_t)s * sendcount + j] = in[s][j];
  return 0;
}

/* ------------------------------------------------------------------------
 * Other element types: IEEE binary16 (fp16) and binary32 (fp32).  The
 * reduction is the same rank-order fp32 accumulation; fp16 is widened
 * exactly and rounded once at the end, fp32 is not rounded at all.
 */

/* fp16 -> fp32, exact.  exponent field e, fraction f (10 bits):
 * e = 0: f * 2^-24 (zero or subnormal); e = 31: inf (f = 0) or NaN;
 * otherwise (1024 + f) * 2^(e - 25). */
float oracle_f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) & 1u;
  const uint32_t e = (uint32_t)(h >> 10) & 0x1Fu;
  const uint32_t f = (uint32_t)h & 0x3FFu;
  float mag;
  if (e == 0u) {
    mag = ldexpf((float)f, -24);
  } else if (e == 31u) {
    uint32_t u = f ? (0x7FC00000u | (f << 13)) : 0x7F800000u;
    memcpy(&mag, &u, sizeof mag);
  } else {
    mag = ldexpf((float)(1024u + f), (int)e - 25);
  }
  return sign ? -mag : mag;
}

/*
 * fp32 -> fp16, IEEE 754 round to nearest, ties to even.
 *
 * A finite fp32 value is M * 2^E with M an integer (the 24-bit significand
 * with its implicit bit, or the 23-bit fraction of a subnormal) and
 * E = max(exponent field, 1) - 150.  fp16 represents multiples of the
 * quantum q = 2^(b - 10) in the binade [2^b, 2^(b+1)) for b >= -14, and of
 * 2^-24 below 2^-14.  The value divided by q is rounded to the nearest
 * integer n, ties to the even one; n is then the fp16 significand: below
 * 2^-14 the encoding is n itself (n = 1024 is exactly the smallest normal),
 * in a normal binade it is ((b + 15) << 10) + n - 1024, and n = 2048 moves
 * to the next binade.  Exponents past 15 give infinity.  NaN becomes a
 * quiet NaN keeping the sign and the top fraction bits.
 */
uint16_t oracle_f32_to_f16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t ef = (u >> 23) & 0xFFu;
  const uint32_t frac = u & 0x7FFFFFu;
  if (ef == 0xFFu) {
    if (frac) return (uint16_t)(sign | 0x7E00u | (frac >> 13));
    return (uint16_t)(sign | 0x7C00u);
  }
  if (ef == 0u && frac == 0u) return sign;
  const uint64_t M = ef ? (uint64_t)(frac | 0x800000u) : (uint64_t)frac;
  const int E = (ef ? (int)ef : 1) - 150;
  /* binade of |x|: position of M's top bit */
  int top = 63;
  while (!((M >> top) & 1u)) --top;
  const int b = top + E;
  const int qexp = b >= -14 ? b - 10 : -24;
  const int shift = qexp - E; /* value / q = M / 2^shift */
  uint64_t n;
  if (shift <= 0) {
    n = M << (-shift);
  } else if (shift >= 64) {
    n = 0;
  } else {
    const uint64_t lo = M & ((1ull << shift) - 1ull);
    const uint64_t half = 1ull << (shift - 1);
    n = M >> shift;
    if (lo > half || (lo == half && (n & 1ull))) n += 1;
  }
  if (b < -14) return (uint16_t)(sign | (uint16_t)n); /* subnormal, or exactly 2^-14 */
  int eb = b;
  if (n == 2048u) {
    n = 1024u;
    eb += 1;
  }
  if (eb > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)(((uint32_t)(eb + 15) << 10) + (uint32_t)(n - 1024u)));
}

void oracle_f32_to_f16_array(const float* x, uint16_t* y, size_t n) {
  for (size_t i = 0; i < n; ++i) y[i] = oracle_f32_to_f16_rne(x[i]);
}

int oracle_allreduce_f16(int R, size_t count, const uint16_t* const* in, uint16_t* const* out) {
  if (R < 1 || R > 64) return -1;
  for (size_t i = 0; i < count; ++i) {
    float acc = oracle_f16_to_f32(in[0][i]);
    for (int r = 1; r < R; ++r) acc = acc + oracle_f16_to_f32(in[r][i]);
    const uint16_t y = oracle_f32_to_f16_rne(acc);
    for (int r = 0; r < R; ++r) out[r][i] = y;
  }
  return 0;
}

int oracle_allreduce_f32(int R, size_t count, const float* const* in, float* const* out) {
  if (R < 1 || R > 64) return -1;
  for (size_t i = 0; i < count; ++i) {
    float acc = in[0][i];
    for (int r = 1; r < R; ++r) acc = acc + in[r][i];
    for (int r = 0; r < R; ++r) out[r][i] = acc;
  }
  return 0;
}
