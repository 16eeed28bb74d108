// Persistent-grid fused Adam/AdamW update for sm_103a.
//
// One launch covers the whole shard.  CTA b walks the items
// [cta_begin[b], cta_begin[b+1]) of a host-balanced work list, so every CTA
// moves about the same number of bytes whatever the tensor sizes.  Per CTA:
//   1. prologue: each param group's scalars are read once (host values for
//      regular plans, device values for capturable ones) and the bias
//      corrections 1 - beta^step are computed once, into shared memory;
//   2. optional inf/nan screen of g*grad_scale over the CTA's items, then a
//      bounded grid barrier (cooperative launch), then the noop flag is read;
//   3. the update: per item, 128-bit streaming loads of p, m, v and g for
//      kUnroll vectors per thread, all issued before any arithmetic, then
//      the element math and 128-bit streaming stores; a scalar loop takes
//      the ragged tail and runs whose pointers are not vector-aligned;
//   4. capturable plans: the last CTA to finish advances each step counter
//      by (noop != 1).
//
// Element math follows "Enhance Distributed Fused Adam (#1794)",
// DistAdamCapturableFunctor::local_step, one IEEE fp32 operation per step
// of the printed expression (__f*_rn intrinsics: correctly rounded and never
// contracted into FMAs), with lerp(beta, a, b) read as beta*b + (1-beta)*a.
// The param-remainder pack and split follow _bf16_rem_to_fp32 of
// "apex/contrib/optimizers/distributed_fused_adam.py" and its inverse.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fadam_internal.h"

namespace fadam {

// Vectors per thread per iteration of the aligned loop.
constexpr int kUnroll = 2;
// Iterations of the grid-barrier wait before it gives up (about a second).
constexpr unsigned kBarrierSpinLimit = 1u << 21;

// ---- scalar state -----------------------------------------------------------

struct SGroup {
  float beta1, omb1, beta2, omb2;  // omb = 1 - beta, rounded once
  float bc1, bc2, eps, wd, lr, gs;
  int32_t step_old;                // counter as read (capturable) or the host step
  uint32_t bits;
};

struct Scal {
  float beta1, omb1, beta2, omb2, bc1, bc2, eps, wd, lr, gs;
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire_s32(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- element types ----------------------------------------------------------

template <int DT> struct Raw4;  // storage of 4 consecutive elements
template <> struct Raw4<FADAM_DT_F32> { using T = float4; };
template <> struct Raw4<FADAM_DT_BF16> { using T = uint2; };
template <> struct Raw4<FADAM_DT_F16> { using T = uint2; };

__device__ __forceinline__ float bf16_to_f32(unsigned short h) {
  return __uint_as_float(static_cast<unsigned>(h) << 16);
}
__device__ __forceinline__ float f16_to_f32(unsigned short h) {
  return __half2float(__ushort_as_half(h));
}

template <int DT>
__device__ __forceinline__ typename Raw4<DT>::T load4(const void* base, int i) {
  return __ldcs(reinterpret_cast<const typename Raw4<DT>::T*>(base) + i);
}

template <int DT>
__device__ __forceinline__ void widen4(const typename Raw4<DT>::T& r, float (&o)[4]) {
  if constexpr (DT == FADAM_DT_F32) {
    o[0] = r.x; o[1] = r.y; o[2] = r.z; o[3] = r.w;
  } else {
    const unsigned short h0 = r.x & 0xFFFFu, h1 = r.x >> 16, h2 = r.y & 0xFFFFu, h3 = r.y >> 16;
    if constexpr (DT == FADAM_DT_BF16) {
      o[0] = bf16_to_f32(h0); o[1] = bf16_to_f32(h1); o[2] = bf16_to_f32(h2); o[3] = bf16_to_f32(h3);
    } else {
      o[0] = f16_to_f32(h0); o[1] = f16_to_f32(h1); o[2] = f16_to_f32(h2); o[3] = f16_to_f32(h3);
    }
  }
}

template <int DT>
__device__ __forceinline__ float load1(const void* base, int i) {
  if constexpr (DT == FADAM_DT_F32) {
    return __ldcs(reinterpret_cast<const float*>(base) + i);
  } else if constexpr (DT == FADAM_DT_BF16) {
    return bf16_to_f32(__ldcs(reinterpret_cast<const unsigned short*>(base) + i));
  } else {
    return f16_to_f32(__ldcs(reinterpret_cast<const unsigned short*>(base) + i));
  }
}

template <int DT>
__device__ __forceinline__ unsigned short narrow(float x) {
  if constexpr (DT == FADAM_DT_BF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  } else {
    return __half_as_ushort(__float2half_rn(x));
  }
}

template <int OT>
__device__ __forceinline__ void store_out4(void* base, int i, const float (&x)[4]) {
  if constexpr (OT == FADAM_DT_F32) {
    __stcs(reinterpret_cast<float4*>(base) + i, make_float4(x[0], x[1], x[2], x[3]));
  } else if constexpr (OT == FADAM_DT_BF16 || OT == FADAM_DT_F16) {
    uint2 w;
    w.x = static_cast<unsigned>(narrow<OT>(x[0])) | (static_cast<unsigned>(narrow<OT>(x[1])) << 16);
    w.y = static_cast<unsigned>(narrow<OT>(x[2])) | (static_cast<unsigned>(narrow<OT>(x[3])) << 16);
    __stcs(reinterpret_cast<uint2*>(base) + i, w);
  }
}

template <int OT>
__device__ __forceinline__ void store_out1(void* base, int i, float x) {
  if constexpr (OT == FADAM_DT_F32) {
    __stcs(reinterpret_cast<float*>(base) + i, x);
  } else if constexpr (OT == FADAM_DT_BF16 || OT == FADAM_DT_F16) {
    __stcs(reinterpret_cast<unsigned short*>(base) + i, narrow<OT>(x));
  }
}

// ---- the update of one element ---------------------------------------------

// p' for the fp32 master x; m and v are updated in place.
template <bool ADAMW>
__device__ __forceinline__ float adam_elem(float x, float& m, float& v, float g, const Scal& s) {
  float sg = __fmul_rn(g, s.gs);
  if constexpr (!ADAMW) sg = __fadd_rn(sg, __fmul_rn(s.wd, x));
  const float sq = __fmul_rn(sg, sg);
  const float m_next = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, sg));
  const float v_next = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.omb2, sq));
  const float m_hat = __fdiv_rn(m_next, s.bc1);
  const float v_hat = __fdiv_rn(v_next, s.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
  float upd = __fdiv_rn(m_hat, denom);
  if constexpr (ADAMW) upd = __fadd_rn(upd, __fmul_rn(s.wd, x));
  m = m_next;
  v = v_next;
  return __fsub_rn(x, __fmul_rn(s.lr, upd));
}

// fp32 master from (bf16 high half, int16 remainder): the high half loses
// the rounding carry when the remainder is negative (16-bit arithmetic).
__device__ __forceinline__ float rem_pack(unsigned short hi, unsigned short rem_bits) {
  const unsigned short h = static_cast<unsigned short>(hi - (rem_bits >> 15));
  return __uint_as_float((static_cast<unsigned>(h) << 16) | rem_bits);
}

// Split an fp32 master into (bf16 high half, int16 remainder bits): the
// high half gains one (mod 2^16) when bit 15 of the low half is set.
__device__ __forceinline__ void rem_split(float x, unsigned short& hi, unsigned short& rem_bits) {
  const unsigned b = __float_as_uint(x);
  rem_bits = static_cast<unsigned short>(b & 0xFFFFu);
  hi = static_cast<unsigned short>((b >> 16) + (rem_bits >> 15));
}

// ---- one work item ------------------------------------------------------------

template <bool ADAMW, int GT, int OT>
__device__ __forceinline__ void run_item_f32(const Item& it, const Scal& s) {
  const int n = it.n;
  int scalar_from = 0;
  if (it.flags & kItemVec) {
    const int nv = n / kVec;
    float4* p4 = reinterpret_cast<float4*>(it.p);
    float4* m4 = reinterpret_cast<float4*>(it.m);
    float4* v4 = reinterpret_cast<float4*>(it.v);
    for (int base = threadIdx.x; base < nv; base += kBlock * kUnroll) {
      float4 P[kUnroll], M[kUnroll], V[kUnroll];
      typename Raw4<GT>::T G[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kBlock;
        if (i < nv) {
          P[u] = __ldcs(p4 + i);
          M[u] = __ldcs(m4 + i);
          V[u] = __ldcs(v4 + i);
          G[u] = load4<GT>(it.g, i);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kBlock;
        if (i < nv) {
          float g[4];
          widen4<GT>(G[u], g);
          float x[4] = {P[u].x, P[u].y, P[u].z, P[u].w};
          float m[4] = {M[u].x, M[u].y, M[u].z, M[u].w};
          float v[4] = {V[u].x, V[u].y, V[u].z, V[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = adam_elem<ADAMW>(x[e], m[e], v[e], g[e], s);
          __stcs(p4 + i, make_float4(x[0], x[1], x[2], x[3]));
          __stcs(m4 + i, make_float4(m[0], m[1], m[2], m[3]));
          __stcs(v4 + i, make_float4(v[0], v[1], v[2], v[3]));
          store_out4<OT>(it.p_out, i, x);
        }
      }
    }
    scalar_from = nv * kVec;
  }
  float* p = reinterpret_cast<float*>(it.p);
  float* mp = reinterpret_cast<float*>(it.m);
  float* vp = reinterpret_cast<float*>(it.v);
  for (int i = scalar_from + threadIdx.x; i < n; i += kBlock) {
    float m = __ldcs(mp + i), v = __ldcs(vp + i);
    const float x = adam_elem<ADAMW>(__ldcs(p + i), m, v, load1<GT>(it.g, i), s);
    __stcs(p + i, x);
    __stcs(mp + i, m);
    __stcs(vp + i, v);
    store_out1<OT>(it.p_out, i, x);
  }
}

// Remainder form: p is the bf16 high half (read), rem the int16 low half
// (read and written), p_out receives the new bf16 high half (it may alias p).
template <bool ADAMW, int GT>
__device__ __forceinline__ void run_item_rem(const Item& it, const Scal& s) {
  const int n = it.n;
  int scalar_from = 0;
  if (it.flags & kItemVec) {
    const int nv = n / kVec;
    const uint2* h4 = reinterpret_cast<const uint2*>(it.p);
    uint2* r4 = reinterpret_cast<uint2*>(it.rem);
    float4* m4 = reinterpret_cast<float4*>(it.m);
    float4* v4 = reinterpret_cast<float4*>(it.v);
    uint2* o4 = reinterpret_cast<uint2*>(it.p_out);
    for (int base = threadIdx.x; base < nv; base += kBlock * kUnroll) {
      uint2 H[kUnroll], R[kUnroll];
      float4 M[kUnroll], V[kUnroll];
      typename Raw4<GT>::T G[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kBlock;
        if (i < nv) {
          H[u] = __ldcs(h4 + i);
          R[u] = __ldcs(r4 + i);
          M[u] = __ldcs(m4 + i);
          V[u] = __ldcs(v4 + i);
          G[u] = load4<GT>(it.g, i);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kBlock;
        if (i < nv) {
          float g[4];
          widen4<GT>(G[u], g);
          const unsigned short hh[4] = {
              static_cast<unsigned short>(H[u].x & 0xFFFFu), static_cast<unsigned short>(H[u].x >> 16),
              static_cast<unsigned short>(H[u].y & 0xFFFFu), static_cast<unsigned short>(H[u].y >> 16)};
          const unsigned short rr[4] = {
              static_cast<unsigned short>(R[u].x & 0xFFFFu), static_cast<unsigned short>(R[u].x >> 16),
              static_cast<unsigned short>(R[u].y & 0xFFFFu), static_cast<unsigned short>(R[u].y >> 16)};
          float m[4] = {M[u].x, M[u].y, M[u].z, M[u].w};
          float v[4] = {V[u].x, V[u].y, V[u].z, V[u].w};
          unsigned short oh[4], orr[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x = adam_elem<ADAMW>(rem_pack(hh[e], rr[e]), m[e], v[e], g[e], s);
            rem_split(x, oh[e], orr[e]);
          }
          __stcs(r4 + i, make_uint2(orr[0] | (static_cast<unsigned>(orr[1]) << 16),
                                    orr[2] | (static_cast<unsigned>(orr[3]) << 16)));
          __stcs(m4 + i, make_float4(m[0], m[1], m[2], m[3]));
          __stcs(v4 + i, make_float4(v[0], v[1], v[2], v[3]));
          __stcs(o4 + i, make_uint2(oh[0] | (static_cast<unsigned>(oh[1]) << 16),
                                    oh[2] | (static_cast<unsigned>(oh[3]) << 16)));
        }
      }
    }
    scalar_from = nv * kVec;
  }
  const unsigned short* hp = reinterpret_cast<const unsigned short*>(it.p);
  unsigned short* rp = reinterpret_cast<unsigned short*>(it.rem);
  float* mp = reinterpret_cast<float*>(it.m);
  float* vp = reinterpret_cast<float*>(it.v);
  unsigned short* op = reinterpret_cast<unsigned short*>(it.p_out);
  for (int i = scalar_from + threadIdx.x; i < n; i += kBlock) {
    float m = __ldcs(mp + i), v = __ldcs(vp + i);
    const float x0 = rem_pack(__ldcs(hp + i), __ldcs(rp + i));
    const float x = adam_elem<ADAMW>(x0, m, v, load1<GT>(it.g, i), s);
    unsigned short oh, orr;
    rem_split(x, oh, orr);
    __stcs(rp + i, orr);
    __stcs(mp + i, m);
    __stcs(vp + i, v);
    __stcs(op + i, oh);
  }
}

// True when this thread saw a non-finite g*grad_scale in the item.
template <int GT>
__device__ __forceinline__ bool scan_item(const Item& it, float gs) {
  bool bad = false;
  const int n = it.n;
  int scalar_from = 0;
  if (it.flags & kItemVec) {
    const int nv = n / kVec;
    for (int i = threadIdx.x; i < nv; i += kBlock) {
      float g[4];
      widen4<GT>(load4<GT>(it.g, i), g);
#pragma unroll
      for (int e = 0; e < 4; ++e) bad |= !isfinite(__fmul_rn(g[e], gs));
    }
    scalar_from = nv * kVec;
  }
  for (int i = scalar_from + threadIdx.x; i < n; i += kBlock)
    bad |= !isfinite(__fmul_rn(load1<GT>(it.g, i), gs));
  return bad;
}

__device__ __forceinline__ Item load_item(const Item* items, int k) {
  const int4* src = reinterpret_cast<const int4*>(items + k);
  int4 w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = __ldg(src + j);
  Item it;
  memcpy(&it, w, sizeof(Item));
  return it;
}

// Grid-wide barrier for a cooperative launch.  The wait is bounded: after
// kBarrierSpinLimit polls it records FADAM_ETIMEOUT in the status block and
// returns false instead of hanging.
__device__ __forceinline__ bool grid_barrier(KScratch* sc) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = ld_acquire_u32(&sc->bar_gen);
    __threadfence();
    const unsigned arrived = atomicAdd(&sc->bar_count, 1u);
    if (arrived == gridDim.x - 1) {
      atomicExch(&sc->bar_count, 0u);
      __threadfence();
      atomicAdd(&sc->bar_gen, 1u);
    } else {
      unsigned spins = 0;
      while (ld_acquire_u32(&sc->bar_gen) == gen) {
        if (++spins > kBarrierSpinLimit) {
          atomicExch(&sc->status, FADAM_ETIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(256);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---- the kernel ---------------------------------------------------------------

template <int GT, int OT, bool REM>
__global__ void __launch_bounds__(kBlock) fadam_update_kernel(const __grid_constant__ KParams kp) {
  __shared__ SGroup sgrp[FADAM_MAX_GROUPS];
  __shared__ int s_noop;
  const bool capturable = (kp.flags & kCapturable) != 0;
  const int tid = threadIdx.x;

  // 1. prologue: scalars once per CTA
  if (tid == 0) s_noop = kp.noop ? (__ldcg(kp.noop) == 1) : 0;  // only 1 means set
  if (tid < kp.n_groups) {
    const KGroup& G = kp.groups[tid];
    SGroup s;
    s.beta1 = G.beta1;
    s.beta2 = G.beta2;
    s.omb1 = __fsub_rn(1.0f, G.beta1);
    s.omb2 = __fsub_rn(1.0f, G.beta2);
    s.eps = G.eps;
    s.wd = G.wd;
    s.bits = G.bits;
    int32_t step;
    if (capturable) {
      s.lr = G.lr_dev ? __ldcg(G.lr_dev) : 0.0f;
      s.gs = G.gs_dev ? __ldcg(G.gs_dev) : 0.0f;
      s.step_old = __ldcg(G.step_dev);
      step = (kp.flags & kPreadvanced) ? s.step_old : s.step_old + 1;
    } else {
      s.lr = G.lr;
      s.gs = G.grad_scale;
      s.step_old = G.step;
      step = G.step;
    }
    if (G.bits & kGroupBiasCorr) {
      s.bc1 = static_cast<float>(1.0 - pow(static_cast<double>(G.beta1), static_cast<double>(step)));
      s.bc2 = static_cast<float>(1.0 - pow(static_cast<double>(G.beta2), static_cast<double>(step)));
    } else {
      s.bc1 = 1.0f;
      s.bc2 = 1.0f;
    }
    sgrp[tid] = s;
  }
  __syncthreads();

  const int item_begin = __ldg(kp.cta_begin + blockIdx.x);
  const int item_end = __ldg(kp.cta_begin + blockIdx.x + 1);
  bool barrier_ok = true;

  // 2. optional inf/nan screen over the whole shard before any update
  if (kp.flags & kCheckFinite) {
    bool bad = false;
    if (!s_noop) {
      for (int k = item_begin; k < item_end; ++k) {
        const Item it = load_item(kp.items, k);
        bad |= scan_item<GT>(it, sgrp[it.group].gs);
      }
    }
    if (__syncthreads_or(bad) && tid == 0) atomicExch(kp.noop, 1);
    barrier_ok = grid_barrier(kp.scratch);
    if (tid == 0) s_noop = (ld_acquire_s32(kp.noop) == 1);
    __syncthreads();
  }

  // 3. the update
  if (!s_noop && barrier_ok) {
    for (int k = item_begin; k < item_end; ++k) {
      const Item it = load_item(kp.items, k);
      const SGroup& G = sgrp[it.group];
      const Scal s{G.beta1, G.omb1, G.beta2, G.omb2, G.bc1, G.bc2, G.eps, G.wd, G.lr, G.gs};
      if constexpr (REM) {
        if (G.bits & kGroupAdamW) run_item_rem<true, GT>(it, s);
        else run_item_rem<false, GT>(it, s);
      } else {
        if (G.bits & kGroupAdamW) run_item_f32<true, GT, OT>(it, s);
        else run_item_f32<false, GT, OT>(it, s);
      }
    }
  }

  // 4. capturable: the last CTA to finish advances the step counters
  if (capturable && !(kp.flags & kPreadvanced)) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(&kp.scratch->done, 1u);
      if (prev == gridDim.x - 1) {
        __threadfence();
        const int adv = (s_noop || !barrier_ok) ? 0 : 1;
        for (int g = 0; g < kp.n_groups; ++g)
          if (sgrp[g].bits & kGroupOwnsStep) *kp.groups[g].step_dev = sgrp[g].step_old + adv;
        atomicExch(&kp.scratch->done, 0u);
      }
    }
  }
}

// Entry for one g dtype: every out dtype, with and without remainders.
template <int GT>
const void* kernel_for(int out_dtype, bool remainders) {
  if (remainders)
    return out_dtype == FADAM_DT_BF16
               ? reinterpret_cast<const void*>(&fadam_update_kernel<GT, FADAM_DT_BF16, true>)
               : nullptr;
  switch (out_dtype) {
    case FADAM_DT_NONE: return reinterpret_cast<const void*>(&fadam_update_kernel<GT, FADAM_DT_NONE, false>);
    case FADAM_DT_F32: return reinterpret_cast<const void*>(&fadam_update_kernel<GT, FADAM_DT_F32, false>);
    case FADAM_DT_BF16: return reinterpret_cast<const void*>(&fadam_update_kernel<GT, FADAM_DT_BF16, false>);
    case FADAM_DT_F16: return reinterpret_cast<const void*>(&fadam_update_kernel<GT, FADAM_DT_F16, false>);
    default: return nullptr;
  }
}

}  // namespace fadam
