/*
 * OpenMP driver that times the oracle on the host cores (the benchmark's
 * CPU baseline and its reference arm).
 *
 * TEST INFRASTRUCTURE ONLY, like fadam_oracle.c, with which it is compiled
 * into a separate, timed-only library (-O3 -fopenmp, vectorisation allowed;
 * -ffp-contract=off kept so that the results stay the oracle's on every
 * host).  The parity library is built from fadam_oracle.c alone, -O2,
 * without OpenMP.
 *
 * It has no arithmetic of its own: each call splits one tensor's elements
 * into one contiguous range per OpenMP thread and calls the oracle's
 * per-tensor function on each range (every element updates independently,
 * so the result is the same as one call over the whole tensor).
 */
#include <omp.h>
#include <stddef.h>
#include <stdint.h>

void oracle_adam_f32(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                     float beta2, float eps, float wd, float lr, float grad_scale, float* p,
                     float* m, float* v, const void* g, int g_dtype, void* p_out, int out_dtype);
void oracle_adam_rem(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                     float beta2, float eps, float wd, float lr, float grad_scale,
                     const uint16_t* p_hi, int16_t* rem, float* m, float* v, const void* g,
                     int g_dtype, uint16_t* p_out);

/* Threads an OpenMP parallel region of this library uses. */
int oracle_omp_threads(void) { return omp_get_max_threads(); }

static size_t elem_bytes(int dtype) { return dtype == 1 ? 4u : dtype == 0 ? 0u : 2u; }

/* oracle_adam_f32 over [0, n), one contiguous range per thread. */
void oracle_omp_adam_f32(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                         float beta2, float eps, float wd, float lr, float grad_scale, float* p,
                         float* m, float* v, const void* g, int g_dtype, void* p_out,
                         int out_dtype) {
#pragma omp parallel
  {
    const int64_t t = omp_get_thread_num(), nt = omp_get_num_threads();
    const int64_t a = n * t / nt, b = n * (t + 1) / nt;
    if (b > a)
      oracle_adam_f32(b - a, mode, bias_correction, step, beta1, beta2, eps, wd, lr, grad_scale,
                      p + a, m + a, v + a, (const char*)g + (size_t)a * elem_bytes(g_dtype),
                      g_dtype, p_out ? (char*)p_out + (size_t)a * elem_bytes(out_dtype) : NULL,
                      out_dtype);
  }
}

/* oracle_adam_rem over [0, n), one contiguous range per thread. */
void oracle_omp_adam_rem(int64_t n, int mode, int bias_correction, int32_t step, float beta1,
                         float beta2, float eps, float wd, float lr, float grad_scale,
                         const uint16_t* p_hi, int16_t* rem, float* m, float* v, const void* g,
                         int g_dtype, uint16_t* p_out) {
#pragma omp parallel
  {
    const int64_t t = omp_get_thread_num(), nt = omp_get_num_threads();
    const int64_t a = n * t / nt, b = n * (t + 1) / nt;
    if (b > a)
      oracle_adam_rem(b - a, mode, bias_correction, step, beta1, beta2, eps, wd, lr, grad_scale,
                      p_hi + a, rem + a, m + a, v + a,
                      (const char*)g + (size_t)a * elem_bytes(g_dtype), g_dtype, p_out + a);
  }
}
