/*
 * Plain CPU oracle for the multi-tensor fused Adam/AdamW shard update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only through the seeded inputs the tests
 * hand to both.
 *
 * What it follows (page titles, then the construct on the page):
 *  - "Enhance Distributed Fused Adam (#1794)" (apex patch),
 *    DistAdamCapturableFunctor: local_step (the L2 branch ADAM_MODE_0 and the
 *    decoupled weight-decay branch), the bias-correction block of operator(),
 *    the early return on the noop flag, and the static_cast of the updated
 *    fp32 parameter to the param-out dtype.
 *  - "apex/contrib/optimizers/distributed_fused_adam.py",
 *    _bf16_rem_to_fp32 (how a bf16 high half and an int16 remainder make the
 *    fp32 master), and the load path of the v2 state dict (the remainder is
 *    the low 16 bits of the fp32 master).
 *
 * Arithmetic: every value the kernel keeps in `float` is a C `float` here,
 * one IEEE operation at a time, in the order the functor states it.  Build
 * with -ffp-contract=off so that no multiply-add is fused.  The readings of
 * points the pages leave open are:
 *  - lerp(beta, a, b) is not defined on the pages; it is read as the Adam
 *    moving average beta*b + (1-beta)*a, two products and one sum.
 *  - pow(beta, step) is evaluated in double and the difference 1 - pow is
 *    rounded to float once.
 *  - The param-out cast to bf16/fp16 rounds to nearest, ties to even.
 *  - The remainder split is the exact inverse of _bf16_rem_to_fp32: the high
 *    half is rounded up in magnitude when bit 15 of the low half is set.
 *
 * Parity pins for each function live in tests/test_oracle_pins.py; every
 * function here is pinned (hand-derived worked examples, closed forms,
 * exhaustive round trips, library conversions), none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_DT_NONE 0
#define ORC_DT_F32 1
#define ORC_DT_BF16 2
#define ORC_DT_F16 3

#define ORC_MODE_L2 0
#define ORC_MODE_ADAMW 1

static uint32_t bits_of(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return u;
}

static float float_of(uint32_t u) {
  float x;
  memcpy(&x, &u, sizeof x);
  return x;
}

/* ---- scalar conversions ------------------------------------------------- */

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
float oracle_bf16_to_f32(uint16_t h) { return float_of((uint32_t)h << 16); }

/* fp16 -> fp32 is exact for every fp16 value, subnormals included. */
float oracle_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t e = ((uint32_t)h >> 10) & 0x1Fu;
  uint32_t f = (uint32_t)h & 0x3FFu;
  if (e == 0) {
    /* subnormal or zero: value = f * 2^-24, exact in float */
    float mag = (float)f * 5.9604644775390625e-08f;
    return sign ? -mag : mag;
  }
  if (e == 31) return float_of(sign | 0x7F800000u | (f << 13));
  return float_of(sign | ((e + 112u) << 23) | (f << 13));
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays a (quiet) NaN. */
uint16_t oracle_f32_to_bf16(float x) {
  uint32_t u = bits_of(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t hi = u >> 16;
  uint32_t lo = u & 0xFFFFu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* fp32 -> fp16, round to nearest, ties to even, with fp16 subnormals and
 * overflow to infinity; NaN stays a (quiet) NaN. */
uint16_t oracle_f32_to_f16(float x) {
  uint32_t u = bits_of(x);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u | ((a >> 13) & 0x3FFu));
  if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 */
  if (a >= 0x38800000u) {                                  /* >= 2^-14: normal */
    uint32_t h = (((a >> 23) - 112u) << 10) | ((a & 0x7FFFFFu) >> 13);
    uint32_t rest = a & 0x1FFFu;
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
  }
  if (a <= 0x33000000u) return (uint16_t)sign; /* <= 2^-25 rounds to zero */
  {
    /* fp16 subnormal: count units of 2^-24 */
    uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126u - (a >> 23); /* 14 .. 24 */
    uint32_t q = mant >> shift;
    uint32_t rest = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rest > half || (rest == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
  }
}

/* ---- param remainders --------------------------------------------------- */

/* _bf16_rem_to_fp32: undo the rounding of the bf16 high half (subtract one
 * when the remainder is negative, in 16-bit arithmetic) and put the
 * remainder in the low half of the fp32 bits. */
uint32_t oracle_rem_pack(uint16_t bf16_bits, int16_t rem) {
  uint16_t hi = (uint16_t)(bf16_bits - (rem < 0 ? 1u : 0u));
  return ((uint32_t)hi << 16) | (uint32_t)(uint16_t)rem;
}

/* Inverse of oracle_rem_pack: the low 16 bits become the remainder, and the
 * high half is bumped by one (wrapping in 16 bits) when the remainder's sign
 * bit is set, so that the packing's subtraction restores it. */
void oracle_rem_split(uint32_t fp32_bits, uint16_t* bf16_bits, int16_t* rem) {
  uint16_t lo = (uint16_t)(fp32_bits & 0xFFFFu);
  uint16_t hi = (uint16_t)(fp32_bits >> 16);
  if (lo & 0x8000u) hi = (uint16_t)(hi + 1u);
  *bf16_bits = hi;
  *rem = (int16_t)lo;
}

void oracle_rem_pack_n(int64_t n, const uint16_t* hi, const int16_t* rem, uint32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_rem_pack(hi[i], rem[i]);
}

void oracle_rem_split_n(int64_t n, const uint32_t* in, uint16_t* hi, int16_t* rem) {
  for (int64_t i = 0; i < n; ++i) oracle_rem_split(in[i], &hi[i], &rem[i]);
}

void oracle_f32_to_bf16_n(int64_t n, const float* x, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}

void oracle_f32_to_f16_n(int64_t n, const float* x, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_bf16_to_f32_n(int64_t n, const uint16_t* h, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(h[i]);
}

void oracle_f16_to_f32_n(int64_t n, const uint16_t* h, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(h[i]);
}

/* ---- the update --------------------------------------------------------- */

/* Bias correction 1 - beta^step (functor's bias_correction == 1 branch). */
float oracle_bias_correction(float beta, int32_t step) {
  return (float)(1.0 - pow((double)beta, (double)step));
}

/* Element i of an array of the given dtype, widened to float (exact). */
static float value_at(const void* a, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_DT_F32: return ((const float*)a)[i];
    case ORC_DT_BF16: return oracle_bf16_to_f32(((const uint16_t*)a)[i]);
    default: return oracle_f16_to_f32(((const uint16_t*)a)[i]);
  }
}

static float grad_at(const void* g, int g_dtype, int64_t i) { return value_at(g, g_dtype, i); }

static void put_out(void* out, int out_dtype, int64_t i, float x) {
  switch (out_dtype) {
    case ORC_DT_F32: ((float*)out)[i] = x; break;
    case ORC_DT_BF16: ((uint16_t*)out)[i] = oracle_f32_to_bf16(x); break;
    case ORC_DT_F16: ((uint16_t*)out)[i] = oracle_f32_to_f16(x); break;
    default: break;
  }
}

/* Moving average read of the pages' lerp(beta, a, b): beta*b + (1-beta)*a. */
static float moving_average(float beta, float fresh, float old) {
  float kept = beta * old;
  float one_minus = 1.0f - beta;
  float added = one_minus * fresh;
  return kept + added;
}

/* One element of local_step, in fp32.  `x` is the fp32 master parameter. */
static float update_one(int mode, float beta1, float beta2, float eps, float wd,
                        float lr, float grad_scale, float bc1, float bc2, float x,
                        float* m, float* v, float grad) {
  float sg = grad * grad_scale;
  if (mode == ORC_MODE_L2) {
    float decay = wd * x;
    sg = sg + decay;
  }
  float sq = sg * sg;
  float m_next = moving_average(beta1, sg, *m);
  float v_next = moving_average(beta2, sq, *v);
  float m_hat = m_next / bc1;
  float v_hat = v_next / bc2;
  float denom = sqrtf(v_hat) + eps;
  float upd = m_hat / denom;
  if (mode == ORC_MODE_ADAMW) {
    float decay = wd * x;
    upd = upd + decay;
  }
  *m = m_next;
  *v = v_next;
  float delta = lr * upd;
  return x - delta;
}

/* One tensor with an fp32 master parameter.  p, m, v are updated in place;
 * p_out (may be NULL when out_dtype is NONE) receives the cast copy. */
void oracle_adam_f32(int64_t n, int mode, int bias_correction, int32_t step,
                     float beta1, float beta2, float eps, float wd, float lr,
                     float grad_scale, float* p, float* m, float* v, const void* g,
                     int g_dtype, void* p_out, int out_dtype) {
  float bc1 = 1.0f, bc2 = 1.0f;
  if (bias_correction == 1) {
    bc1 = oracle_bias_correction(beta1, step);
    bc2 = oracle_bias_correction(beta2, step);
  }
  for (int64_t i = 0; i < n; ++i) {
    float x = update_one(mode, beta1, beta2, eps, wd, lr, grad_scale, bc1, bc2, p[i],
                         &m[i], &v[i], grad_at(g, g_dtype, i));
    p[i] = x;
    if (p_out) put_out(p_out, out_dtype, i, x);
  }
}

/* One tensor whose master and moments are all of `state_dtype` (fp32,
 * bf16 or fp16), as the functor's one type T for p, m and v: each value is
 * widened to float, the update runs in float as above, and p, m, v are
 * rounded back to the state dtype (to nearest, ties to even) when stored.
 * p_out receives the float result cast to its own dtype. */
void oracle_adam_state(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                       float beta2, float eps, float wd, float lr, float grad_scale, void* p,
                       void* m, void* v, int state_dtype, const void* g, int g_dtype,
                       void* p_out, int out_dtype) {
  float bc1 = 1.0f, bc2 = 1.0f;
  if (bias_correction == 1) {
    bc1 = oracle_bias_correction(beta1, step);
    bc2 = oracle_bias_correction(beta2, step);
  }
  for (int64_t i = 0; i < n; ++i) {
    float mi = value_at(m, state_dtype, i);
    float vi = value_at(v, state_dtype, i);
    float x = update_one(mode, beta1, beta2, eps, wd, lr, grad_scale, bc1, bc2,
                         value_at(p, state_dtype, i), &mi, &vi, grad_at(g, g_dtype, i));
    put_out(p, state_dtype, i, x);
    put_out(m, state_dtype, i, mi);
    put_out(v, state_dtype, i, vi);
    if (p_out) put_out(p_out, out_dtype, i, x);
  }
}

/* One tensor with an fp32 master and moments of `moment_dtype` (bf16 or
 * fp16): TransformerEngine's FusedAdam exp_avg_dtype and exp_avg_sq_dtype
 * (constructor arguments of the "[Performance] FusedAdam capturable kernel"
 * issue's adam_bench.py), taken equal.  m and v are widened to float, the
 * update runs in float as above, p keeps the float result and m, v are
 * rounded back to their dtype (to nearest, ties to even) when stored. */
void oracle_adam_moments(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                         float beta2, float eps, float wd, float lr, float grad_scale, float* p,
                         void* m, void* v, int moment_dtype, const void* g, int g_dtype,
                         void* p_out, int out_dtype) {
  float bc1 = 1.0f, bc2 = 1.0f;
  if (bias_correction == 1) {
    bc1 = oracle_bias_correction(beta1, step);
    bc2 = oracle_bias_correction(beta2, step);
  }
  for (int64_t i = 0; i < n; ++i) {
    float mi = value_at(m, moment_dtype, i);
    float vi = value_at(v, moment_dtype, i);
    float x = update_one(mode, beta1, beta2, eps, wd, lr, grad_scale, bc1, bc2, p[i], &mi, &vi,
                         grad_at(g, g_dtype, i));
    p[i] = x;
    put_out(m, moment_dtype, i, mi);
    put_out(v, moment_dtype, i, vi);
    if (p_out) put_out(p_out, out_dtype, i, x);
  }
}

/* One tensor whose fp32 master is held as a bf16 high half plus an int16
 * remainder.  p_hi is read (it is not written unless p_out aliases it),
 * rem, m and v are updated in place, p_out (bf16 bits) gets the new high
 * half. */
void oracle_adam_rem(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                     float beta2, float eps, float wd, float lr, float grad_scale,
                     const uint16_t* p_hi, int16_t* rem, float* m, float* v,
                     const void* g, int g_dtype, uint16_t* p_out) {
  float bc1 = 1.0f, bc2 = 1.0f;
  if (bias_correction == 1) {
    bc1 = oracle_bias_correction(beta1, step);
    bc2 = oracle_bias_correction(beta2, step);
  }
  for (int64_t i = 0; i < n; ++i) {
    float x = float_of(oracle_rem_pack(p_hi[i], rem[i]));
    x = update_one(mode, beta1, beta2, eps, wd, lr, grad_scale, bc1, bc2, x, &m[i], &v[i],
                   grad_at(g, g_dtype, i));
    uint16_t hi;
    int16_t r;
    oracle_rem_split(bits_of(x), &hi, &r);
    rem[i] = r;
    p_out[i] = hi;
  }
}

/* The same update carried out in double, for error analysis only: the
 * inputs and hyper-parameters are the float values widened to double and
 * nothing is rounded to float along the way. */
void oracle_adam_f64(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                     float beta2, float eps, float wd, float lr, float grad_scale,
                     double* p, double* m, double* v, const double* g) {
  double b1 = beta1, b2 = beta2, e = eps, w = wd, a = lr, s = grad_scale;
  double bc1 = 1.0, bc2 = 1.0;
  if (bias_correction == 1) {
    bc1 = 1.0 - pow(b1, (double)step);
    bc2 = 1.0 - pow(b2, (double)step);
  }
  for (int64_t i = 0; i < n; ++i) {
    double x = p[i];
    double sg = g[i] * s;
    if (mode == ORC_MODE_L2) sg = sg + w * x;
    double m_next = b1 * m[i] + (1.0 - b1) * sg;
    double v_next = b2 * v[i] + (1.0 - b2) * (sg * sg);
    double upd = (m_next / bc1) / (sqrt(v_next / bc2) + e);
    if (mode == ORC_MODE_ADAMW) upd = upd + w * x;
    m[i] = m_next;
    v[i] = v_next;
    p[i] = x - a * upd;
  }
}

/* Sum of squares of a gradient tensor, each element widened exactly and
 * squared and added in double, one after the other. */
double oracle_sumsq(int64_t n, const void* g, int g_dtype) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double x = (double)grad_at(g, g_dtype, i);
    s += x * x;
  }
  return s;
}

/* Inf/NaN screen of a gradient tensor: 1 when some grad*grad_scale (the
 * scaled gradient the update would consume) is not finite, else 0. */
int oracle_any_nonfinite(int64_t n, const void* g, int g_dtype, float grad_scale) {
  for (int64_t i = 0; i < n; ++i) {
    float sg = grad_at(g, g_dtype, i) * grad_scale;
    if (!isfinite(sg)) return 1;
  }
  return 0;
}
