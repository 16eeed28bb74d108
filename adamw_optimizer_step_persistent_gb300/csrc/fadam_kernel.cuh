// Persistent-grid fused Adam/AdamW update for sm_103a.
//
// One launch covers the whole shard.  CTA b walks the items
// [cta_begin[b], cta_begin[b+1]) of a host-balanced work list, so every CTA
// moves about the same number of bytes whatever the tensor sizes.  Per CTA:
//   1. prologue: each param group's scalars are read once (host values for
//      regular plans, device values for capturable ones) and the bias
//      corrections 1 - beta^step are computed once, into shared memory;
//   2. optional inf/nan screen of g*grad_scale over the CTA's items (the
//      same two passes, copying only g), then a bounded grid barrier
//      (cooperative launch), then the noop flag is read;
//   3. the update, in two passes.  The bulk pass treats every
//      16-byte-aligned item as tiles of kTile 4-element vectors, grouped in
//      chunks of up to kChunkTiles tiles that the CTAs pull from one
//      launch-wide counter (so an SM that gets more bandwidth takes more
//      chunks).  In each CTA thread 0 copies the tiles of p, m, v, g (and
//      the remainders) into shared memory with cp.async.bulk, 2-3 tiles
//      ahead and across chunk boundaries, each tile completing on its own
//      mbarrier; every thread updates one vector of the tile from shared
//      memory and writes the results straight to global memory with
//      streaming 128-bit stores.  A tail pass then takes the at most 7
//      trailing elements of every bulk item (warps pull 32 items at a time
//      from another counter, one item per lane), and the rest pass the
//      CTA's statically assigned items that are not 16-byte aligned, with
//      the whole CTA (128-bit streaming loads, then element by element);
//   4. the last CTA to finish resets the work counters and, for capturable
//      plans, advances each step counter by (noop != 1).
//
// p, m and v share one state dtype ST (fp32, bf16 or fp16; the functor's one
// type T), widened to float for the update and rounded back (nearest-even)
// when stored; the remainder form keeps fp32 m and v.
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

#include <type_traits>

#include "fadam_internal.h"

namespace fadam {

// Vectors per thread per iteration of the 128-bit load loop.
#ifndef FADAM_UNROLL
#define FADAM_UNROLL 1
#endif
constexpr int kUnroll = FADAM_UNROLL;
// Resident CTAs per SM the register allocation must allow (unset: let the
// compiler choose; an explicit 1 changes its choice).
#ifdef FADAM_MIN_BLOCKS
#define FADAM_BOUNDS __launch_bounds__(kBlock, FADAM_MIN_BLOCKS)
#else
#define FADAM_BOUNDS __launch_bounds__(kBlock)
#endif
// Wall time after which a grid-barrier or mbarrier wait gives up.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- scalar state -----------------------------------------------------------

// One group's scalars in shared memory, read by every tile.  Twelve words,
// 16-byte aligned, so that a tile loads the ten it needs with three 128-bit
// loads (a 52-byte record, with no provable vector alignment, took ten
// 32-bit loads per warp and tile: 1-2 % of the 16-bit forms' instructions).
// What the tiles do not read lives in the array after it.
struct alignas(16) SGroup {
  float beta1, omb1, beta2, omb2;  // omb = 1 - beta, rounded once
  float bc1, bc2, eps, wd;
  float lr, gs;
  int32_t step_old;                // counter as read (capturable) or the host step
  uint32_t bits;
};
static_assert(sizeof(SGroup) == 48, "SGroup is three 16-byte words");
// Per group: the step this launch applies.
__shared__ int32_t s_group_step[FADAM_MAX_GROUPS];

// Step counters advance modulo 2^32, as an int32 tensor's += does (no
// signed overflow in the kernel's own arithmetic).
__device__ __forceinline__ int32_t step_add(int32_t a, int32_t b) {
  return static_cast<int32_t>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
}

// 1 - beta^step in double, rounded once to float.
__device__ __forceinline__ float bias_correction(float beta, int32_t step) {
  return static_cast<float>(1.0 - pow(static_cast<double>(beta), static_cast<double>(step)));
}

// The memo entry of group g for `step`, if it holds that step's corrections
// for these betas.
__device__ __forceinline__ bool memo_lookup(const BcMemo* memo, int g, float beta1, float beta2,
                                            int32_t step, float& bc1, float& bc2) {
  const BcMemo* e = memo + 2 * g + (step & 1);
  const uint4 a = __ldcg(reinterpret_cast<const uint4*>(e));
  const uint4 b = __ldcg(reinterpret_cast<const uint4*>(e) + 1);
  if (a.w != kMemoTag || a.x != __float_as_uint(beta1) || a.y != __float_as_uint(beta2) ||
      static_cast<int32_t>(a.z) != step)
    return false;
  bc1 = __uint_as_float(b.x);
  bc2 = __uint_as_float(b.y);
  return true;
}

// Group g's corrections for `step` into its memo entry (the other parity's
// entry than the one this launch reads).
__device__ __forceinline__ void memo_store(BcMemo* memo, int g, float beta1, float beta2,
                                           int32_t step) {
  BcMemo* e = memo + 2 * g + (step & 1);
  const uint4 b = make_uint4(__float_as_uint(bias_correction(beta1, step)),
                             __float_as_uint(bias_correction(beta2, step)), 0u, 0u);
  const uint4 a = make_uint4(__float_as_uint(beta1), __float_as_uint(beta2),
                             static_cast<unsigned>(step), kMemoTag);
  __stcg(reinterpret_cast<uint4*>(e) + 1, b);
  __stcg(reinterpret_cast<uint4*>(e), a);
}

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
  } else if constexpr (DT == FADAM_DT_BF16) {
    // a bf16 is the top half of its float: one shift or one mask per value
    o[0] = __uint_as_float(r.x << 16); o[1] = __uint_as_float(r.x & 0xFFFF0000u);
    o[2] = __uint_as_float(r.y << 16); o[3] = __uint_as_float(r.y & 0xFFFF0000u);
  } else {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
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

// Two floats rounded to dtype DT (nearest-even) in one 32-bit word, the
// first in the low half: one paired conversion instead of two and a pack.
template <int DT>
__device__ __forceinline__ unsigned narrow2(float lo, float hi) {
  if constexpr (DT == FADAM_DT_BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const unsigned*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const unsigned*>(&h);
  }
}

// 4 floats rounded to dtype DT (nearest-even for 16-bit types).
template <int DT>
__device__ __forceinline__ typename Raw4<DT>::T pack_out4(const float (&x)[4]) {
  if constexpr (DT == FADAM_DT_F32) {
    return make_float4(x[0], x[1], x[2], x[3]);
  } else {
    return make_uint2(narrow2<DT>(x[0], x[1]), narrow2<DT>(x[2], x[3]));
  }
}

// Extra destinations of the param-out copy (the all-gather side of the
// data-parallel exchange): the same element lands at the same byte offset
// from each destination's start as from p_out's.
struct Dests {
  int n;
  const int64_t* delta;
};

template <class T>
__device__ __forceinline__ void store_all(T* base, int i, const T& x, const Dests* d) {
  __stcs(base + i, x);
  if (d)
    for (int k = 0; k < d->n; ++k)
      __stcs(reinterpret_cast<T*>(reinterpret_cast<char*>(base) + d->delta[k]) + i, x);
}

template <int OT>
__device__ __forceinline__ void store_out4(void* base, int i, const float (&x)[4],
                                           const Dests* d = nullptr) {
  if constexpr (OT == FADAM_DT_F32 || OT == FADAM_DT_BF16 || OT == FADAM_DT_F16)
    store_all(reinterpret_cast<typename Raw4<OT>::T*>(base), i, pack_out4<OT>(x), d);
}

template <int OT>
__device__ __forceinline__ void store_out1(void* base, int i, float x, const Dests* d = nullptr) {
  if constexpr (OT == FADAM_DT_F32) {
    store_all(reinterpret_cast<float*>(base), i, x, d);
  } else if constexpr (OT == FADAM_DT_BF16 || OT == FADAM_DT_F16) {
    store_all(reinterpret_cast<unsigned short*>(base), i, narrow<OT>(x), d);
  }
}

__device__ __forceinline__ void unpack4(const uint2& r, unsigned short (&o)[4]) {
  o[0] = static_cast<unsigned short>(r.x & 0xFFFFu);
  o[1] = static_cast<unsigned short>(r.x >> 16);
  o[2] = static_cast<unsigned short>(r.y & 0xFFFFu);
  o[3] = static_cast<unsigned short>(r.y >> 16);
}

__device__ __forceinline__ uint2 pack4(const unsigned short (&h)[4]) {
  return make_uint2(h[0] | (static_cast<unsigned>(h[1]) << 16), h[2] | (static_cast<unsigned>(h[3]) << 16));
}

// What a pipeline pass moves through shared memory.
// kScan: only g, for the inf/nan screen; kNorm: only g, for the squared norm;
// kReduce: the exchange sources' slices of g, reduced into the shard's g;
// kScaledA / kScaledB: the two update passes of a scaled 16-bit state (A
// writes param-out and takes each tensor's absmax of the new values, B
// stores the rescaled state).
enum class Pass { kUpdate, kScan, kNorm, kReduce, kScaledA, kScaledB };

__host__ __device__ constexpr bool update_like(Pass p) {
  return p == Pass::kUpdate || p == Pass::kScaledA || p == Pass::kScaledB;
}

// A scaled tensor's factors for one pass: the stored scales of p, m, v
// (to unscale) and, in the rescale pass, the reciprocals of the new ones.
struct StateScale {
  float s[3];
  float r[3];
};

// Scaled state, absmax slots: 1 + the largest |x| bit pattern seen (NaN's
// patterns sort above inf's, so a NaN wins as it does in a min/max scan;
// 0 means no element seen).
__device__ __forceinline__ unsigned abs_bits(float x) { return __float_as_uint(x) & 0x7fffffffu; }

// ---- the update of one element ---------------------------------------------

// Bias corrections equal to 1 in float: with bias correction off, and once
// beta^step has fallen below half an ulp of 1 (from step 165 for beta 0.9,
// 338 for 0.95, 17,321 for 0.999), the division by the correction is
// an IEEE identity.  A UNIT mask names the divisions an instance leaves out;
// the result is the same bits either way.  kRecipBc (FADAM_RECIP_BC) turns
// the remaining divisions by bc1 and bc2 into products with their
// reciprocals, which the caller then passes in place of bc1 and bc2: a
// second rounding, within the tolerance, not the same bits.
enum : int { kUnitBc1 = 1, kUnitBc2 = 2, kRecipBc = 4 };

// p' for the fp32 master x; m and v are updated in place.
template <bool ADAMW, int UNIT = 0>
__device__ __forceinline__ float adam_elem(float x, float& m, float& v, float g, const Scal& s) {
  float sg = __fmul_rn(g, s.gs);
  if constexpr (!ADAMW) sg = __fadd_rn(sg, __fmul_rn(s.wd, x));
  const float sq = __fmul_rn(sg, sg);
  const float m_next = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, sg));
  const float v_next = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.omb2, sq));
  float m_hat = m_next, v_hat = v_next;
  if constexpr (UNIT & kRecipBc) {  // s.bc1, s.bc2 hold the reciprocals
    if constexpr (!(UNIT & kUnitBc1)) m_hat = __fmul_rn(m_next, s.bc1);
    if constexpr (!(UNIT & kUnitBc2)) v_hat = __fmul_rn(v_next, s.bc2);
  } else {
    if constexpr (!(UNIT & kUnitBc1)) m_hat = __fdiv_rn(m_next, s.bc1);
    if constexpr (!(UNIT & kUnitBc2)) v_hat = __fdiv_rn(v_next, s.bc2);
  }
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

// One 4-element vector whose p, m, v have dtype ST, in registers: widened
// to float, updated, rounded back to ST (nearest-even) when stored.
// Scaled state (PASS kScaledA / kScaledB): the widened values are first
// multiplied by the tensor's scales; pass A then writes only param-out and
// folds |p'|, |m'|, |v'| into the thread's maxima `mx` (bit patterns), pass
// B only the state, each new value times its new reciprocal scale.
template <bool ADAMW, int ST, int GT, int OT, Pass PASS = Pass::kUpdate, int UNIT = 0>
__device__ __forceinline__ void update4_state(const typename Raw4<p_dtype_of(ST)>::T& P,
                                              const typename Raw4<mv_dtype_of(ST)>::T& M,
                                              const typename Raw4<mv_dtype_of(ST)>::T& V,
                                              const typename Raw4<GT>::T& G, const Scal& s, void* p,
                                              void* m, void* v, void* out, int i, const Dests& d,
                                              const StateScale* sc = nullptr,
                                              unsigned* mx = nullptr) {
  float g[4], x[4], mm[4], vv[4];
  widen4<GT>(G, g);
  constexpr int PT = p_dtype_of(ST), MT = mv_dtype_of(ST);
  widen4<PT>(P, x);
  widen4<MT>(M, mm);
  widen4<MT>(V, vv);
  if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = __fmul_rn(x[e], sc->s[0]);
      mm[e] = __fmul_rn(mm[e], sc->s[1]);
      vv[e] = __fmul_rn(vv[e], sc->s[2]);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = adam_elem<ADAMW, UNIT>(x[e], mm[e], vv[e], g[e], s);
  if constexpr (PASS == Pass::kScaledA) {
    store_out4<OT>(out, i, x, &d);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx[0] = max(mx[0], abs_bits(x[e]));
      mx[1] = max(mx[1], abs_bits(mm[e]));
      mx[2] = max(mx[2], abs_bits(vv[e]));
    }
  } else if constexpr (PASS == Pass::kScaledB) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = __fmul_rn(x[e], sc->r[0]);
      mm[e] = __fmul_rn(mm[e], sc->r[1]);
      vv[e] = __fmul_rn(vv[e], sc->r[2]);
    }
    store_out4<PT>(p, i, x);
    store_out4<MT>(m, i, mm);
    store_out4<MT>(v, i, vv);
  } else {
    store_out4<PT>(p, i, x);
    store_out4<MT>(m, i, mm);
    store_out4<MT>(v, i, vv);
    store_out4<OT>(out, i, x, &d);
  }
}

// Pass A, items off the tiles (the rest pass, a CTA at a time): a warp's
// maxima into the tensor's absmax slots (1 + bits).
__device__ __forceinline__ void flush_absmax(const KParams& kp, int t, unsigned (&mx)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const unsigned w = __reduce_max_sync(0xffffffffu, mx[k]);
    if ((threadIdx.x & 31) == 0) atomicMax(kp.absmax + 3 * t + k, w + 1u);
    mx[k] = 0u;
  }
}

// Pass A, bulk tiles: a warp's maxima into the CTA's shared slots (1 + bits,
// 0 = none yet); thread 0 takes them to the tensor's global slots with
// push_absmax once every warp has added its own.
__device__ __forceinline__ void gather_absmax(unsigned* sm, unsigned (&mx)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const unsigned w = __reduce_max_sync(0xffffffffu, mx[k]);
    if ((threadIdx.x & 31) == 0) atomicMax(sm + k, w + 1u);
    mx[k] = 0u;
  }
}

// Thread 0: the CTA's maxima of tensor t into its global slots, and the
// shared slots cleared for a later item.
__device__ __forceinline__ void push_absmax(const KParams& kp, int t, unsigned* sm) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const unsigned a = sm[k];
    if (a) atomicMax(kp.absmax + 3 * t + k, a);
    sm[k] = 0u;
  }
}

// One 4-element vector of the remainder form: H the bf16 high halves, R the
// remainders; the new remainders go to rem, the new high halves to out.
template <bool ADAMW, int GT>
__device__ __forceinline__ void update4_rem(const uint2& H, const uint2& R, float4 M, float4 V,
                                            const typename Raw4<GT>::T& G, const Scal& s,
                                            uint2* r4, float4* m4, float4* v4, uint2* o4, int i,
                                            const Dests& d) {
  float g[4];
  widen4<GT>(G, g);
  unsigned short hh[4], rr[4], oh[4], orr[4];
  unpack4(H, hh);
  unpack4(R, rr);
  float m[4] = {M.x, M.y, M.z, M.w};
  float v[4] = {V.x, V.y, V.z, V.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x = adam_elem<ADAMW>(rem_pack(hh[e], rr[e]), m[e], v[e], g[e], s);
    rem_split(x, oh[e], orr[e]);
  }
  __stcs(r4 + i, pack4(orr));
  __stcs(m4 + i, make_float4(m[0], m[1], m[2], m[3]));
  __stcs(v4 + i, make_float4(v[0], v[1], v[2], v[3]));
  store_all(o4, i, pack4(oh), &d);
}

// ---- bulk-copy pipeline -----------------------------------------------------

#ifndef FADAM_BULK
#define FADAM_BULK 1
#endif
// Tiles in flight per CTA: up to kMaxStages, as many as fit in
// kStageBudget bytes of dynamic shared memory (at least two).  Three 64 KB
// stages and the static shared memory fit the 227 KB a CTA may use; with
// one 1024-thread CTA per SM (the register file allows no second one) that
// space would otherwise sit idle.  Layouts with larger tiles keep two.
#ifndef FADAM_STAGES
#define FADAM_STAGES 3
#endif
constexpr int kMaxStages = FADAM_STAGES;
constexpr unsigned kStageBudget = 192u * 1024u;
constexpr int kTile = kBlock;  // vectors per tile: one per thread

// Vectors of one tile a thread has in flight at once (the tile loop's unroll).
#ifndef FADAM_VEC_UNROLL
#define FADAM_VEC_UNROLL 2
#endif
constexpr int kVecUnroll = FADAM_VEC_UNROLL;

template <int DT>
__host__ __device__ constexpr int vec_bytes() { return DT == FADAM_DT_F32 ? 16 : 8; }

// Byte layout of one update tile in shared memory, stream after stream, for
// p, m, v of dtype ST (or, in remainder form, the bf16 high halves and the
// int16 remainders with fp32 m and v) and g of dtype GT.
template <int ST, int GT, bool REM>
struct Layout {
  static constexpr int kP = REM ? 8 : vec_bytes<p_dtype_of(ST)>();  // bytes per vector of p
  static constexpr int kR = REM ? 8 : 0;                  // ... of the remainders
  static constexpr int kMV = REM ? 16 : vec_bytes<mv_dtype_of(ST)>();  // ... of m and of v
  static constexpr int kG = vec_bytes<GT>();              // ... of g
  static constexpr unsigned per_vector = kP + kR + 2 * kMV + kG;
  // vectors of an update tile: two per thread when a vector carries at most
  // 40 bytes (16-bit state), so every tile keeps about 64 KB in flight
  static constexpr int update_vectors = (per_vector <= 40 ? 2 : 1) * kTile;
  static constexpr int off_r = kP * update_vectors;
  static constexpr int off_m = (kP + kR) * update_vectors;
  static constexpr int off_v = off_m + kMV * update_vectors;
  static constexpr int off_g = off_v + kMV * update_vectors;
  static constexpr unsigned update_tile = per_vector * update_vectors;
  // the g-only passes (screen, norm, reduce) fill a stage of at least
  // 64 KB with g: four vectors per thread for fp32 grads, eight for 16-bit
  // ones (more when the update's tile is larger)
  static constexpr unsigned kScanBytes = 65536u;
  static constexpr unsigned scan_target = update_tile > kScanBytes ? update_tile : kScanBytes;
  static constexpr int scan_per_thread = static_cast<int>(scan_target / kG / kTile);
  static constexpr int scan_vectors = scan_per_thread * kTile;
  static constexpr unsigned scan_tile = scan_vectors * kG;
  static constexpr unsigned stage = update_tile > scan_tile ? update_tile : scan_tile;
  // buffers of the pipeline that fit the budget (at least two)
  static constexpr int stages = kStageBudget / stage >= unsigned(kMaxStages) ? kMaxStages : 2;
};

// Pipeline buffers of one kernel instance; every pass of an instance uses
// the same count, so the stage counter carries from pass to pass.  The
// scaled-state instances keep two: their spilled registers live in L1,
// which shares the SM's memory with these buffers, and a third 64 KB stage
// cost them more than it gained.
template <int ST, int GT, bool REM, bool SCALED>
__host__ __device__ constexpr int pipeline_stages() {
  return SCALED ? 2 : Layout<ST, GT, REM>::stages;
}

template <int ST, int GT, bool REM, bool SCALED = false>
__host__ __device__ constexpr size_t smem_bytes() {
  return FADAM_BULK ? size_t(pipeline_stages<ST, GT, REM, SCALED>()) * Layout<ST, GT, REM>::stage : 0;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `parity` to complete, for at most kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// Global -> shared bulk copy completing on `bar` (16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
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

// Vectors of an item that go through the bulk pipeline: all of them when
// every stream is 16-byte aligned, rounded down to an even count so that
// 8-byte-per-vector streams still copy whole 16-byte units; none otherwise.
__device__ __forceinline__ int bulk_vectors(const Item& it) {
  return (it.flags & kItemBulk) ? ((it.n / kVec) & ~1) : 0;
}

__device__ __forceinline__ int bulk_tiles(const Item& it) {
  return (bulk_vectors(it) + kTile - 1) / kTile;
}


// Vectors of a reduce tile: as many as the R source slices (and, when
// accumulating, the shard's own g as one slice more) fit in one stage (at
// most as many as a screen tile), a multiple of one warp.
template <int ST, int GT, bool REM>
__host__ __device__ constexpr int reduce_vectors(int n_sources) {
  using L = Layout<ST, GT, REM>;
  const int v = static_cast<int>(L::stage / (static_cast<unsigned>(n_sources) * L::kG));
  return (v < L::scan_vectors ? v : L::scan_vectors) & ~31;
}

// Slices a reduce tile copies: the sources, and the shard's own g when
// accumulating.
__device__ __forceinline__ int reduce_slices(const KParams& kp) {
  return kp.n_sources + ((kp.average & kExchangeAccumulate) ? 1 : 0);
}

// Vectors in one tile of a pass (Layout::update_vectors or ::scan_vectors).
template <int ST, int GT, bool REM, Pass PASS>
__host__ __device__ constexpr int tile_vectors() {
  return update_like(PASS) ? Layout<ST, GT, REM>::update_vectors
                               : Layout<ST, GT, REM>::scan_vectors;
}

// Thread 0 of the CTA: start the copies of vectors [v0, v0 + len) of `it`
// into buffer `slot % NS` (NS: the instance's pipeline stages).
template <int ST, int GT, bool REM, Pass PASS, int NS>
__device__ __forceinline__ void issue_tile(const KParams& kp, const Item& it, int v0, unsigned len,
                                           unsigned slot, unsigned char* smem, uint64_t* full) {
  using L = Layout<ST, GT, REM>;
  const unsigned b = slot % NS;
  unsigned char* st = smem + size_t(b) * L::stage;
  uint64_t* bar = full + b;
  const size_t v = static_cast<size_t>(v0);
  if constexpr (PASS == Pass::kReduce) {
    // source r's slice at r * (vectors of a reduce tile) in the stage; when
    // accumulating, the shard's old g after them
    const int ns = reduce_slices(kp);
    const size_t stride = size_t(reduce_vectors<ST, GT, REM>(ns)) * L::kG;
    mbar_expect_tx(bar, static_cast<unsigned>(ns) * len * L::kG);
    const char* g = static_cast<const char*>(it.g) + v * L::kG;
    for (int r = 0; r < kp.n_sources; ++r)
      bulk_load(st + size_t(r) * stride, g + kp.src_delta[r], len * L::kG, bar);
    if (ns > kp.n_sources) bulk_load(st + size_t(kp.n_sources) * stride, g, len * L::kG, bar);
  } else if constexpr (!update_like(PASS)) {
    mbar_expect_tx(bar, len * L::kG);
    bulk_load(st, static_cast<const char*>(it.g) + v * L::kG, len * L::kG, bar);
  } else {
    mbar_expect_tx(bar, len * L::per_vector);
    bulk_load(st, static_cast<const char*>(it.p) + v * L::kP, len * L::kP, bar);
    if constexpr (REM)
      bulk_load(st + L::off_r, reinterpret_cast<const char*>(it.rem) + v * L::kR, len * L::kR, bar);
    bulk_load(st + L::off_m, static_cast<const char*>(it.m) + v * L::kMV, len * L::kMV, bar);
    bulk_load(st + L::off_v, static_cast<const char*>(it.v) + v * L::kMV, len * L::kMV, bar);
    bulk_load(st + L::off_g, static_cast<const char*>(it.g) + v * L::kG, len * L::kG, bar);
  }
}

// The producer side of the pipeline, kept by thread 0 only: it pulls chunks
// of tiles from the launch-wide counter (so faster SMs take more of them)
// and copies their tiles Layout::stages ahead of the consumers, announcing each
// tile's (item, tile) in a small shared ring before its copies start.  When
// the chunks run out it announces the end with an arrival that carries no
// bytes.  The g-only passes take chunks in batches of consecutive indices,
// up to kBatchMax while much work remains and down to one near the end (so
// the CTAs still finish together); a batch's chunk records arrive in one
// round trip.
constexpr int kBatchMax = 8;


struct Producer {
  Item it;
  Chunk recs[kBatchMax];  // the current batch's chunk records
  StateScale sc;          // scaled-state passes: the current item's factors
  int item, v, vend;      // vectors [v, vend) of the current chunk remain
  int chunk;
  int next, batch0, batch_end;  // chunks [next, batch_end) of the batch remain
  unsigned slot;
  bool finished;
};

struct TileTag {
  int item;  // -1: no more tiles
  int v0;
  int len;
  int chunk;
  StateScale sc;  // scaled-state passes only
};

// The factors of tensor t: the stored scales, and for the rescale pass the
// reciprocal of each new scale (absmax / target; the reciprocal only where
// the scale is positive, else 0).  Read after the grid barrier that
// follows the absmax pass.
__device__ __forceinline__ StateScale tensor_scales(const KParams& kp, int t, bool rescale) {
  StateScale sc;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    sc.s[k] = __ldcg(kp.scales + 3 * t + k);
    sc.r[k] = 0.0f;
    if (rescale) {
      const unsigned a = __ldcg(kp.absmax + 3 * t + k);
      const float scale = a ? __fdiv_rn(__uint_as_float(a - 1u), kp.max_scaled) : 0.0f;
      sc.r[k] = scale > 0.0f ? __fdiv_rn(1.0f, scale) : 0.0f;
    }
  }
  return sc;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Thread 0: take the next batch of chunks, or return false when none is left.
__device__ __forceinline__ bool next_batch(Producer& pr, const KParams& kp, unsigned* counter,
                                           int kmax) {
  const int remaining = kp.n_chunks - pr.batch_end;  // as this CTA last saw it
  const int k = max(1, min(kmax, remaining / (2 * static_cast<int>(gridDim.x))));
  const unsigned c0 = atomicAdd(counter, static_cast<unsigned>(k));
  if (c0 >= static_cast<unsigned>(kp.n_chunks)) return false;
  const int cnt = min(k, kp.n_chunks - static_cast<int>(c0));
  for (int j = 0; j < cnt; ++j)  // independent 16-byte copies, one wait
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_addr(&pr.recs[j])),
                 "l"(kp.chunks + c0 + j)
                 : "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  pr.next = static_cast<int>(c0);
  pr.batch0 = static_cast<int>(c0);
  pr.batch_end = static_cast<int>(c0) + cnt;
  return true;
}

template <int ST, int GT, bool REM, Pass PASS, int NS>
__device__ __forceinline__ void produce_next(Producer& pr, const KParams& kp, unsigned* counter,
                                             unsigned char* smem, uint64_t* full, TileTag* tags) {
  if (pr.finished) return;
  while (pr.v >= pr.vend) {
    // the update's chunks are long (16 tiles): one at a time keeps the
    // CTAs on neighbouring chunks; the g-only passes' chunks are 2-4 tiles
    if (pr.next >= pr.batch_end &&
        !next_batch(pr, kp, counter, update_like(PASS) ? 1 : kBatchMax)) {
      const unsigned b = pr.slot % NS;
      tags[b] = TileTag{-1, 0, 0, -1};
      mbar_arrive(full + b);  // completes the phase with no copy
      ++pr.slot;
      pr.finished = true;
      return;
    }
    const Chunk ch = pr.recs[pr.next - pr.batch0];
    pr.chunk = pr.next++;
    if (ch.item != pr.item) {
      pr.item = ch.item;
      pr.it = load_item(kp.items, ch.item);
      if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB)
        pr.sc = tensor_scales(kp, pr.it.tensor, PASS == Pass::kScaledB);
    }
    pr.v = ch.tile0 * kTile;
    pr.vend = min((ch.tile0 + ch.ntiles) * kTile, bulk_vectors(pr.it));
  }
  int tv;
  if constexpr (PASS == Pass::kReduce) tv = reduce_vectors<ST, GT, REM>(reduce_slices(kp));
  else tv = tile_vectors<ST, GT, REM, PASS>();
  const int len = min(tv, pr.vend - pr.v);
  TileTag& tg = tags[pr.slot % NS];
  tg.item = pr.item;
  tg.v0 = pr.v;
  tg.len = len;
  tg.chunk = pr.chunk;
  if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) tg.sc = pr.sc;
  issue_tile<ST, GT, REM, PASS, NS>(kp, pr.it, pr.v, static_cast<unsigned>(len), pr.slot, smem, full);
  pr.v += len;
  ++pr.slot;
}

// Consume one tile from shared memory: thread t takes vectors t, t + kTile,
// ... of it.  DESTS: param-out also goes to the exchange destinations (a
// separate instance, so the plain step carries no destination loop).
template <bool ADAMW, int ST, int GT, int OT, bool REM, bool DESTS, Pass PASS = Pass::kUpdate,
          int UNIT = 0>
__device__ __forceinline__ void update_tile(const Item& it, const Scal& s, const unsigned char* st,
                                            int v0, int len, const Dests& d0,
                                            const StateScale* sc = nullptr, unsigned* mx = nullptr) {
  const Dests d{DESTS ? d0.n : 0, d0.delta};
  using L = Layout<ST, GT, REM>;
  // the scaled passes take their vectors one at a time: interleaving two
  // spills more of their larger working set than it hides
  constexpr int kU = (PASS == Pass::kScaledA || PASS == Pass::kScaledB) ? 1 : kVecUnroll;
#pragma unroll kU
  for (int q = 0; q < L::update_vectors / kTile; ++q) {
    const int t = threadIdx.x + q * kTile;
    if (t >= len) return;
    const int i = v0 + t;
    const typename Raw4<GT>::T G = reinterpret_cast<const typename Raw4<GT>::T*>(st + L::off_g)[t];
    if constexpr (REM) {
      const uint2 H = reinterpret_cast<const uint2*>(st)[t];
      const uint2 R = reinterpret_cast<const uint2*>(st + L::off_r)[t];
      const float4 M = reinterpret_cast<const float4*>(st + L::off_m)[t];
      const float4 V = reinterpret_cast<const float4*>(st + L::off_v)[t];
      update4_rem<ADAMW, GT>(H, R, M, V, G, s, reinterpret_cast<uint2*>(it.rem),
                             reinterpret_cast<float4*>(it.m), reinterpret_cast<float4*>(it.v),
                             reinterpret_cast<uint2*>(it.p_out), i, d);
    } else {
      using P4 = typename Raw4<p_dtype_of(ST)>::T;
      using M4 = typename Raw4<mv_dtype_of(ST)>::T;
      const P4 P = reinterpret_cast<const P4*>(st)[t];
      const M4 M = reinterpret_cast<const M4*>(st + L::off_m)[t];
      const M4 V = reinterpret_cast<const M4*>(st + L::off_v)[t];
      update4_state<ADAMW, ST, GT, OT, PASS, UNIT>(P, M, V, G, s, it.p, it.m, it.v, it.p_out, i,
                                                   d, sc, mx);
    }
  }
}

// The 16-bit state forms are bound by instruction issue, not by memory:
// their update passes have instances without the divisions by bias
// corrections equal to 1 in every group (a launch-wide choice, so that each
// instance is a loop of its own).  Every other form keeps one instance (its
// divisions issue within the memory time).
template <int ST, bool REM>
__host__ __device__ constexpr bool unit_bc_instances() {
  return !REM && (ST == FADAM_DT_BF16 || ST == FADAM_DT_F16);
}



// ---- the reduce-scatter stand-in ---------------------------------------------
//
// "apex/contrib/optimizers/distributed_fused_adam.py", _start_bucket_grad_sync:
// this rank's shard of g from the R ranks' contributions, widened to float
// and added in rank order (one IEEE addition each), divided by R for
// ReduceOp.AVG (one IEEE division), rounded once to the grad dtype.
// Accumulating (_finish_bucket_grad_sync's grads_shard.add_ after the first
// reduce-scatter of a step), that rounded value is added to the shard's old
// g, both widened, and the sum rounded once more.  With the screen on, the
// new g*grad_scale is tested as the update will use it.

template <int GT>
__device__ __forceinline__ float stored_value(float x) {
  if constexpr (GT == FADAM_DT_F32) return x;
  else if constexpr (GT == FADAM_DT_BF16) return bf16_to_f32(narrow<GT>(x));
  else return f16_to_f32(narrow<GT>(x));
}

// One tile: source r's vectors at r * stride in the stage (ACC: the
// shard's old g after them).  R > 0: the number of sources, fixed at
// compile time (the source loop unrolled, the slice offsets constants);
// R == 0: kp.n_sources.  Either way the sources are added in rank order.
template <int ST, int GT, bool REM, int R, bool ACC>
__device__ __forceinline__ bool reduce_tile(const KParams& kp, const Item& it,
                                            const unsigned char* st, int v0, int len, float gs,
                                            bool screen) {
  using L = Layout<ST, GT, REM>;
  using G4 = typename Raw4<GT>::T;
  const int nr = R > 0 ? R : kp.n_sources;
  const size_t stride = size_t(reduce_vectors<ST, GT, REM>(nr + (ACC ? 1 : 0))) * L::kG;
  const float rn = static_cast<float>(nr);
  bool bad = false;
  for (int t = threadIdx.x; t < len; t += kBlock) {
    float acc[4];
    widen4<GT>(reinterpret_cast<const G4*>(st)[t], acc);
#pragma unroll
    for (int r = 1; r < (R > 0 ? R : FADAM_MAX_SOURCES); ++r) {
      if (R == 0 && r >= nr) break;
      float x[4];
      widen4<GT>(reinterpret_cast<const G4*>(st + size_t(r) * stride)[t], x);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
    }
    if (kp.average & kExchangeAverage) {
      // dividing by a power of two is multiplying by its exact reciprocal
      // (the same correctly rounded result)
      if (kp.avg_mul != 0.0f) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = __fmul_rn(acc[e], kp.avg_mul);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = __fdiv_rn(acc[e], rn);
      }
    }
    if constexpr (ACC) {  // the shard's old g, staged after the sources
      float old[4];
      widen4<GT>(reinterpret_cast<const G4*>(st + size_t(nr) * stride)[t], old);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(old[e], stored_value<GT>(acc[e]));
    }
    const G4 w = pack_out4<GT>(acc);
    __stcs(reinterpret_cast<G4*>(const_cast<void*>(it.g)) + v0 + t, w);
    if (screen) {
      float y[4];
      widen4<GT>(w, y);
#pragma unroll
      for (int e = 0; e < 4; ++e) bad |= !isfinite(__fmul_rn(y[e], gs));
    }
  }
  return bad;
}

// The reduce tile for the launch's source count: common data-parallel
// degrees get an unrolled instance, any other count the generic loop.
template <int ST, int GT, bool REM>
__device__ __forceinline__ bool reduce_tile_any(const KParams& kp, const Item& it,
                                                const unsigned char* st, int v0, int len, float gs,
                                                bool screen) {
  if (kp.average & kExchangeAccumulate) {
    switch (kp.n_sources) {
      case 2: return reduce_tile<ST, GT, REM, 2, true>(kp, it, st, v0, len, gs, screen);
      case 4: return reduce_tile<ST, GT, REM, 4, true>(kp, it, st, v0, len, gs, screen);
      case 8: return reduce_tile<ST, GT, REM, 8, true>(kp, it, st, v0, len, gs, screen);
      default: return reduce_tile<ST, GT, REM, 0, true>(kp, it, st, v0, len, gs, screen);
    }
  }
  switch (kp.n_sources) {
    case 2: return reduce_tile<ST, GT, REM, 2, false>(kp, it, st, v0, len, gs, screen);
    case 4: return reduce_tile<ST, GT, REM, 4, false>(kp, it, st, v0, len, gs, screen);
    case 8: return reduce_tile<ST, GT, REM, 8, false>(kp, it, st, v0, len, gs, screen);
    default: return reduce_tile<ST, GT, REM, 0, false>(kp, it, st, v0, len, gs, screen);
  }
}

// One element, straight from global memory (tails, unaligned items).
template <int GT>
__device__ __forceinline__ bool reduce_elem(const KParams& kp, const Item& it, int i, float gs,
                                            bool screen) {
  const char* g = static_cast<const char*>(it.g);
  float acc = load1<GT>(g + kp.src_delta[0], i);
  for (int r = 1; r < kp.n_sources; ++r) acc = __fadd_rn(acc, load1<GT>(g + kp.src_delta[r], i));
  if (kp.average & kExchangeAverage)
    acc = kp.avg_mul != 0.0f ? __fmul_rn(acc, kp.avg_mul)
                             : __fdiv_rn(acc, static_cast<float>(kp.n_sources));
  if (kp.average & kExchangeAccumulate) acc = __fadd_rn(load1<GT>(g, i), stored_value<GT>(acc));
  store_out1<GT>(const_cast<void*>(it.g), i, acc);
  return screen && !isfinite(__fmul_rn(stored_value<GT>(acc), gs));
}

template <int Q, int GT>
__device__ __forceinline__ bool scan_tile(const unsigned char* st, int len, float gs) {
  bool bad = false;
#pragma unroll
  for (int q = 0; q < Q; ++q) {  // Q = Layout::scan_per_thread
    const int t = threadIdx.x + q * kTile;
    if (t < len) {
      float g[4];
      widen4<GT>(reinterpret_cast<const typename Raw4<GT>::T*>(st)[t], g);
#pragma unroll
      for (int e = 0; e < 4; ++e) bad |= !isfinite(__fmul_rn(g[e], gs));
    }
  }
  return bad;
}

// OR of the raw words of 4 elements (zero only when every element is +0).
template <int DT>
__device__ __forceinline__ unsigned raw_or4(const typename Raw4<DT>::T& r) {
  if constexpr (DT == FADAM_DT_F32)
    return __float_as_uint(r.x) | __float_as_uint(r.y) | __float_as_uint(r.z) | __float_as_uint(r.w);
  else
    return r.x | r.y;
}

// Sum of the squares of 4 widened values in float.  `special` is set when
// that sum is outside the range where float serves (overflow, NaN, or
// nonzero values whose squares underflow); such vectors are redone exactly
// in double by square_tile_exact.
__device__ __forceinline__ float square4(const float (&g)[4], bool& special) {
  const float v = __fadd_rn(__fadd_rn(__fmul_rn(g[0], g[0]), __fmul_rn(g[1], g[1])),
                            __fadd_rn(__fmul_rn(g[2], g[2]), __fmul_rn(g[3], g[3])));
  const bool tiny_nonzero = v < 1e-30f && (g[0] != 0.0f || g[1] != 0.0f || g[2] != 0.0f || g[3] != 0.0f);
  special |= !(v <= 1e30f) || tiny_nonzero;
  return v;
}

struct SqPart {
  float f;
  double d;
};

// The rare case, kept out of line so that no double arithmetic sits in the
// streaming loop: the thread's vectors of one tile again, the in-range ones
// summed in float as before and the others squared exactly in double.
template <int Q, int GT>
__device__ __noinline__ SqPart square_tile_exact(const unsigned char* st, int len) {
  SqPart r{0.0f, 0.0};
  for (int q = 0; q < Q; ++q) {
    const int t = threadIdx.x + q * kTile;
    if (t < len) {
      float g[4];
      widen4<GT>(reinterpret_cast<const typename Raw4<GT>::T*>(st)[t], g);
      bool sp = false;
      const float v = square4(g, sp);
      if (sp) {
        for (int e = 0; e < 4; ++e) r.d += static_cast<double>(g[e]) * static_cast<double>(g[e]);
      } else {
        r.f = __fadd_rn(r.f, v);
      }
    }
  }
  return r;
}

// A thread's running sum of squares over the tiles of one chunk: float with
// Kahan compensation, in registers, plus a double part for the rare values
// square4 sends there (and for float sums that grow large).  The double
// part lives in shared memory (one slot per thread, `has_d` says it is
// nonzero), so the out-of-line code that touches it takes no reference to
// the registers.  At the end of a chunk the CTA reduces all threads' sums in
// a fixed order into the chunk's slot, so the result does not depend on
// which CTA took which chunk.
struct NormAcc {
  float sum, comp;
  bool has_d;
  int chunk;
  int group;
};

static __device__ __noinline__ float2 norm_fold(float sum, float comp, double d, double* dpart) {
  double x = *dpart + d;
  if (sum > 1e30f) {  // keep the float part far from overflow
    x += static_cast<double>(sum) - static_cast<double>(comp);
    sum = 0.0f;
    comp = 0.0f;
  }
  *dpart = x;
  return make_float2(sum, comp);
}

__device__ __forceinline__ void norm_add(NormAcc& na, float f, double d, bool special,
                                         double* dpart) {
  const float y = __fsub_rn(f, na.comp);
  const float t = __fadd_rn(na.sum, y);
  na.comp = __fsub_rn(__fsub_rn(t, na.sum), y);
  na.sum = t;
  if (special || na.sum > 1e30f) {
    const float2 sc = norm_fold(na.sum, na.comp, d, dpart);
    na.sum = sc.x;
    na.comp = sc.y;
    na.has_d = true;
  }
}

// Sum of one double per thread over the whole CTA, in a fixed order; the
// result is valid in thread 0.  Every thread must call it.
__device__ __forceinline__ double cta_sum(double x, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = x;
  __syncthreads();
  double total = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kBlock / 32; ++w) total += red[w];
  __syncthreads();  // red is reused
  return total;
}

// The per-chunk reduction rides on the bulk pipeline's one CTA barrier per
// tile.  When a chunk ends, each warp reduces its threads' float sums in
// float (five roundings) into f[warp] of one of two buffers, and its double
// parts into d[warp] (zero unless some thread of the warp holds one); after
// the next barrier warp 0 adds the 32 warp partials, again in float and in
// a fixed order, and folds in the double parts and grad_scale^2 in double,
// into the chunk's slot.  Every partial is a sum of squares (nonnegative),
// so each of these roundings adds at most 2^-24 of the chunk's sum.  The
// double arithmetic stays with one thread per chunk: this GPU's FP64 rate
// is a small fraction of its FP32 rate, and 32 warps converting and adding
// in double at every close held the whole CTA at the next barrier.  The
// buffers alternate, so a chunk that ends in the following tile writes the
// other one while warp 0 still reads.  The result does not depend on which
// CTA took which chunk.
struct NormPending {
  int chunk;  // -1: nothing to publish
  float gs;
};

struct NormBuf {
  float* f;
  double* d;
};

// Buffer k % 2 of the warp partials in `red` (3 * kBlock / 32 doubles: the
// two double halves, then the two float halves).
__device__ __forceinline__ NormBuf norm_buf(double* red, unsigned k) {
  constexpr int W = kBlock / 32;
  return NormBuf{reinterpret_cast<float*>(red + 2 * W) + (k & 1u) * W, red + (k & 1u) * W};
}

__device__ __forceinline__ void norm_warp_close(NormAcc& na, const NormBuf& buf, double* dpart) {
  float xf = na.sum;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) xf = __fadd_rn(xf, __shfl_xor_sync(0xffffffffu, xf, o));
  double xd = 0.0;
  if (__any_sync(0xffffffffu, na.has_d)) {
    if (na.has_d) {
      xd = *dpart;
      *dpart = 0.0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xd += __shfl_xor_sync(0xffffffffu, xd, o);
  }
  if ((threadIdx.x & 31) == 0) {
    buf.f[threadIdx.x / 32] = xf;
    buf.d[threadIdx.x / 32] = xd;
  }
  na.sum = 0.0f;
  na.comp = 0.0f;
  na.has_d = false;
}

// Warp 0, after a CTA barrier that follows every warp's norm_warp_close.
__device__ __forceinline__ void norm_publish(const NormBuf& buf, float gs, double* slot) {
  constexpr int W = kBlock / 32;  // warp partials (lanes past them add zeros)
  if (threadIdx.x < 32) {
    float y = threadIdx.x < W ? buf.f[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) y = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, o));
    double yd = threadIdx.x < W ? buf.d[threadIdx.x] : 0.0;
    if (__any_sync(0xffffffffu, __double_as_longlong(yd) != 0)) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) yd += __shfl_xor_sync(0xffffffffu, yd, o);
    }
    // thread 0 writes every chunk slot; its fence before the completion
    // count at the end of the launch publishes them all
    if (threadIdx.x == 0) *slot = static_cast<double>(gs) * gs * (static_cast<double>(y) + yd);
  }
}

// Every thread of the CTA calls this for the same tile (the warp-level
// close needs whole warps).  A chunk that ends here becomes `pend`.
template <int Q, int GT>
__device__ __forceinline__ void norm_tile(const unsigned char* st, const TileTag& tag, int group,
                                          NormAcc& na, const SGroup* sgrp, double* red,
                                          double* dpart, unsigned& closes, NormPending& pend) {
  if (tag.chunk != na.chunk) {
    if (na.chunk >= 0) {
      norm_warp_close(na, norm_buf(red, closes), dpart);
      pend = NormPending{na.chunk, sgrp[na.group].gs};
      ++closes;
    }
    na.chunk = tag.chunk;
    na.group = group;
  }
  // Squares summed with fused multiply-adds in two independent chains (the
  // thread's even and odd vectors), added once per tile; full tiles skip
  // the per-vector bounds test.  The range test is made once on the
  // thread's tile sum: overflow or NaN, or a tiny sum while some input is
  // nonzero (squares that may have underflowed; the raw words are OR-ed
  // and the sign bits masked off).  Either sends the thread's vectors of
  // this tile to the exact path.
  using R4 = typename Raw4<GT>::T;
  const R4* src = reinterpret_cast<const R4*>(st);
  float f2[2] = {0.0f, 0.0f};
  unsigned nz = 0u;
  if (tag.len == Q * kTile) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {  // Q = Layout::scan_per_thread
      const R4 r = src[threadIdx.x + q * kTile];
      float g[4];
      widen4<GT>(r, g);
#pragma unroll
      for (int e = 0; e < 4; ++e) f2[q & 1] = __fmaf_rn(g[e], g[e], f2[q & 1]);
      nz |= raw_or4<GT>(r);
    }
  } else {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int t = threadIdx.x + q * kTile;
      if (t < tag.len) {
        const R4 r = src[t];
        float g[4];
        widen4<GT>(r, g);
#pragma unroll
        for (int e = 0; e < 4; ++e) f2[q & 1] = __fmaf_rn(g[e], g[e], f2[q & 1]);
        nz |= raw_or4<GT>(r);
      }
    }
  }
  float f = __fadd_rn(f2[0], f2[1]);
  const unsigned mag = GT == FADAM_DT_F32 ? 0x7fffffffu : 0x7fff7fffu;
  const bool special = !(f <= 1e30f) || (f < 1e-30f && (nz & mag) != 0u);
  double d = 0.0;
  if (special) {
    const SqPart r = square_tile_exact<Q, GT>(st, tag.len);
    f = r.f;
    d = r.d;
  }
  norm_add(na, f, d, special, dpart);
}

// Phase A: the bulk tiles of the whole shard, pulled chunk by chunk from
// the launch-wide counter, as one continuous pipeline per CTA (the copies
// of the next chunk start while the current one is consumed).  `bad`
// collects the scan's finding; a wait that gives up sets `timed_out` and
// ends the pass for the CTA.
template <int ST, int GT, int OT, bool REM, Pass PASS, int NS, int UNIT = 0>
__device__ __forceinline__ void bulk_pass(const KParams& kp, const SGroup* sgrp, unsigned* counter,
                                          unsigned char* smem, uint64_t* full, TileTag* tags,
                                          Producer& pr, double* red, unsigned& stage, bool& bad,
                                          bool& timed_out) {
  const Dests dst{kp.n_dests, kp.dst_delta};
  const bool screen = (kp.flags & kCheckFinite) != 0;  // reduce pass: screen the result
  unsigned mx[3] = {0u, 0u, 0u};                        // scaled pass A: |new value| maxima
  // scaled pass A: when the tiles move on to another item, the warps' maxima
  // of the one they leave meet in shared memory and thread 0 takes them to
  // the global slots after the tile's barrier (three global atomics per CTA
  // and item, not three per warp: with 152 CTAs on neighbouring chunks of
  // one tensor, those land on the same three words).  Two buffers: the
  // warps may fill the next one while thread 0 empties the last.
  __shared__ unsigned s_amax[2][3];
  int amax_tensor = -1;  // tensor whose maxima wait in s_amax[amax_buf ^ 1]
  unsigned amax_buf = 0;  // the buffer the next gather fills
  if constexpr (PASS == Pass::kScaledA) {
    if (threadIdx.x < 6) s_amax[threadIdx.x / 3][threadIdx.x % 3] = 0u;  // read after a tile's barrier
  }
  NormAcc na{0.0f, 0.0f, false, -1, 0};
  NormPending pend{-1, 0.0f};
  double* dpart = nullptr;
  if constexpr (PASS == Pass::kNorm) {
    __shared__ double s_dpart[kBlock];
    dpart = s_dpart + threadIdx.x;
    *dpart = 0.0;
  }
  unsigned closes = 0;
  if (threadIdx.x == 0) {
    pr.item = -1;
    pr.v = 0;
    pr.vend = 0;
    pr.slot = stage;
    pr.finished = false;
    pr.next = pr.batch0 = pr.batch_end = 0;
    for (int q = 0; q < NS; ++q) produce_next<ST, GT, REM, PASS, NS>(pr, kp, counter, smem, full, tags);
  }
  int cur_item = -1;
  Item it;
  for (;; ++stage) {
    const unsigned b = stage % NS;
    bool ok = mbar_wait(full + b, (stage / NS) & 1u);
    // the norm's chunk closes and the absmax flushes are warp-wide: one
    // decision per warp
    if constexpr (PASS == Pass::kNorm || PASS == Pass::kScaledA) ok = __all_sync(0xffffffffu, ok);
    TileTag tag{-1, 0, 0, -1};
    if (ok) {
      tag = tags[b];
      if (tag.item >= 0) {
        if (tag.item != cur_item) {
          if constexpr (PASS == Pass::kScaledA) {
            if (cur_item >= 0) {
              gather_absmax(s_amax[amax_buf], mx);
              amax_tensor = it.tensor;
              amax_buf ^= 1u;
            }
          }
          cur_item = tag.item;
          it = load_item(kp.items, tag.item);
        }
        const unsigned char* st = smem + size_t(b) * Layout<ST, GT, REM>::stage;
        const SGroup& G = sgrp[it.group];
        const Scal s{G.beta1, G.omb1, G.beta2, G.omb2, G.bc1, G.bc2, G.eps, G.wd, G.lr, G.gs};
        if constexpr (PASS == Pass::kScan) {
          bad |= scan_tile<Layout<ST, GT, REM>::scan_per_thread, GT>(st, tag.len, s.gs);
        } else if constexpr (PASS == Pass::kNorm) {
          norm_tile<Layout<ST, GT, REM>::scan_per_thread, GT>(st, tag, it.group, na, sgrp, red,
                                                              dpart, closes, pend);
        } else if constexpr (PASS == Pass::kReduce) {
          bad |= reduce_tile_any<ST, GT, REM>(kp, it, st, tag.v0, tag.len, s.gs, screen);
        } else if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) {
          const StateScale sc = tag.sc;
          if (G.bits & kGroupAdamW)
            update_tile<true, ST, GT, OT, REM, true, PASS, UNIT>(it, s, st, tag.v0, tag.len, dst,
                                                                 &sc, mx);
          else
            update_tile<false, ST, GT, OT, REM, true, PASS, UNIT>(it, s, st, tag.v0, tag.len, dst,
                                                                  &sc, mx);
        } else {
          const bool aw = (G.bits & kGroupAdamW) != 0;
          constexpr Pass U = Pass::kUpdate;
          if (dst.n == 0) {
            if (aw) update_tile<true, ST, GT, OT, REM, false, U, UNIT>(it, s, st, tag.v0, tag.len, dst);
            else update_tile<false, ST, GT, OT, REM, false, U, UNIT>(it, s, st, tag.v0, tag.len, dst);
          } else {
            if (aw) update_tile<true, ST, GT, OT, REM, true, U, UNIT>(it, s, st, tag.v0, tag.len, dst);
            else update_tile<false, ST, GT, OT, REM, true, U, UNIT>(it, s, st, tag.v0, tag.len, dst);
          }
        }
      }
    }
    // every thread is done with buffer b; a timeout anywhere stops the CTA
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      ++stage;
      return;
    }
    if constexpr (PASS == Pass::kNorm) {
      if (pend.chunk >= 0) {
        norm_publish(norm_buf(red, closes - 1u), pend.gs, kp.partials + pend.chunk);
        pend.chunk = -1;
      }
    }
    if constexpr (PASS == Pass::kScaledA) {
      if (amax_tensor >= 0) {  // every warp's gather came before the barrier
        if (threadIdx.x == 0) push_absmax(kp, amax_tensor, s_amax[amax_buf ^ 1u]);
        amax_tensor = -1;
      }
    }
    if (tag.item < 0) {  // the end marker (the same for every thread)
      ++stage;
      if constexpr (PASS == Pass::kScaledA) {
        if (cur_item >= 0) {
          gather_absmax(s_amax[amax_buf], mx);
          __syncthreads();
          if (threadIdx.x == 0) push_absmax(kp, it.tensor, s_amax[amax_buf]);
        }
      }
      if constexpr (PASS == Pass::kNorm) {
        if (na.chunk >= 0) {
          const NormBuf buf = norm_buf(red, closes);
          norm_warp_close(na, buf, dpart);
          __syncthreads();
          norm_publish(buf, sgrp[na.group].gs, kp.partials + na.chunk);
        }
      }
      return;
    }
    if (threadIdx.x == 0) {
      // order the generic-proxy reads of the buffer before its async refill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      produce_next<ST, GT, REM, PASS, NS>(pr, kp, counter, smem, full, tags);
    }
  }
}

// ---- element-wise paths (tails, runs not 16-byte aligned) -------------------

template <bool ADAMW, int ST, int GT, int OT, Pass PASS, int UNIT = 0>
__device__ __forceinline__ void update_elem_state(const Item& it, const Scal& s, int i,
                                                  const Dests& d, const StateScale* sc,
                                                  unsigned* mx) {
  constexpr int PT = p_dtype_of(ST), MT = mv_dtype_of(ST);
  float m = load1<MT>(it.m, i), v = load1<MT>(it.v, i), x0 = load1<PT>(it.p, i);
  if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) {
    x0 = __fmul_rn(x0, sc->s[0]);
    m = __fmul_rn(m, sc->s[1]);
    v = __fmul_rn(v, sc->s[2]);
  }
  const float x = adam_elem<ADAMW, UNIT>(x0, m, v, load1<GT>(it.g, i), s);
  if constexpr (PASS == Pass::kScaledA) {
    store_out1<OT>(it.p_out, i, x, &d);
    mx[0] = max(mx[0], abs_bits(x));
    mx[1] = max(mx[1], abs_bits(m));
    mx[2] = max(mx[2], abs_bits(v));
  } else if constexpr (PASS == Pass::kScaledB) {
    store_out1<PT>(it.p, i, __fmul_rn(x, sc->r[0]));
    store_out1<MT>(it.m, i, __fmul_rn(m, sc->r[1]));
    store_out1<MT>(it.v, i, __fmul_rn(v, sc->r[2]));
  } else {
    store_out1<PT>(it.p, i, x);
    store_out1<MT>(it.m, i, m);
    store_out1<MT>(it.v, i, v);
    store_out1<OT>(it.p_out, i, x, &d);
  }
}

template <bool ADAMW, int GT>
__device__ __forceinline__ void update_elem_rem(const Item& it, const Scal& s, int i,
                                                const Dests& d) {
  const unsigned short* hp = reinterpret_cast<const unsigned short*>(it.p);
  unsigned short* rp = reinterpret_cast<unsigned short*>(it.rem);
  float* mp = reinterpret_cast<float*>(it.m);
  float* vp = reinterpret_cast<float*>(it.v);
  unsigned short* op = reinterpret_cast<unsigned short*>(it.p_out);
  float m = __ldcs(mp + i), v = __ldcs(vp + i);
  const float x0 = rem_pack(__ldcs(hp + i), __ldcs(rp + i));
  const float x = adam_elem<ADAMW>(x0, m, v, load1<GT>(it.g, i), s);
  unsigned short oh, orr;
  rem_split(x, oh, orr);
  __stcs(rp + i, orr);
  __stcs(mp + i, m);
  __stcs(vp + i, v);
  store_all(op, i, oh, &d);
}

template <bool ADAMW, int ST, int GT, int OT, bool REM, Pass PASS = Pass::kUpdate, int UNIT = 0>
__device__ __forceinline__ void update_elem(const Item& it, const Scal& s, int i, const Dests& d,
                                            const StateScale* sc = nullptr, unsigned* mx = nullptr) {
  if constexpr (REM) update_elem_rem<ADAMW, GT>(it, s, i, d);
  else update_elem_state<ADAMW, ST, GT, OT, PASS, UNIT>(it, s, i, d, sc, mx);
}

// A whole item not aligned for bulk copies, by the whole CTA: 128-bit
// streaming loads when every stream is vector-aligned, then element by
// element for the rest.
template <bool ADAMW, int ST, int GT, int OT, bool REM, Pass PASS = Pass::kUpdate, int UNIT = 0>
__device__ __forceinline__ void simt_item(const Item& it, const Scal& s, const Dests& d,
                                          const StateScale* sc = nullptr, unsigned* mx = nullptr) {
  const int n = it.n;
  int scalar_from = 0;
  if (it.flags & kItemVec) {
    const int nv = n / kVec;
    for (int base = threadIdx.x; base < nv; base += kBlock * kUnroll) {
      if constexpr (REM) {
        const uint2* h4 = reinterpret_cast<const uint2*>(it.p);
        uint2* r4 = reinterpret_cast<uint2*>(it.rem);
        float4* m4 = reinterpret_cast<float4*>(it.m);
        float4* v4 = reinterpret_cast<float4*>(it.v);
        uint2* o4 = reinterpret_cast<uint2*>(it.p_out);
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
          if (i < nv) update4_rem<ADAMW, GT>(H[u], R[u], M[u], V[u], G[u], s, r4, m4, v4, o4, i, d);
        }
      } else {
        typename Raw4<p_dtype_of(ST)>::T P[kUnroll];
        typename Raw4<mv_dtype_of(ST)>::T M[kUnroll], V[kUnroll];
        typename Raw4<GT>::T G[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = base + u * kBlock;
          if (i < nv) {
            P[u] = load4<p_dtype_of(ST)>(it.p, i);
            M[u] = load4<mv_dtype_of(ST)>(it.m, i);
            V[u] = load4<mv_dtype_of(ST)>(it.v, i);
            G[u] = load4<GT>(it.g, i);
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = base + u * kBlock;
          if (i < nv)
            update4_state<ADAMW, ST, GT, OT, PASS, UNIT>(P[u], M[u], V[u], G[u], s, it.p, it.m,
                                                         it.v, it.p_out, i, d, sc, mx);
        }
      }
    }
    scalar_from = nv * kVec;
  }
  for (int i = scalar_from + threadIdx.x; i < n; i += kBlock)
    update_elem<ADAMW, ST, GT, OT, REM, PASS, UNIT>(it, s, i, d, sc, mx);
}

// True when this thread saw a non-finite g*grad_scale in the item (by the
// whole CTA).
template <int GT>
__device__ __forceinline__ bool simt_scan(const Item& it, float gs) {
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

// Phase B, tails: the at most 7 trailing elements of every bulk item.
// Warps pull 32 items at a time from a launch-wide counter and each lane
// takes one item's tail, so the many small latencies overlap across the
// whole GPU.
template <int ST, int GT, int OT, bool REM, Pass PASS, int UNIT = 0>
__device__ __forceinline__ bool tail_pass(const KParams& kp, const SGroup* sgrp, unsigned* counter,
                                          int n_items) {
  const int lane = threadIdx.x % 32;
  const Dests dst{kp.n_dests, kp.dst_delta};
  const bool screen = (kp.flags & kCheckFinite) != 0;
  bool bad = false;
  for (;;) {
    unsigned base = 0;
    if (lane == 0) base = atomicAdd(counter, 32u);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (base >= static_cast<unsigned>(n_items)) break;
    const int k = static_cast<int>(base) + lane;
    if (k >= n_items) continue;
    const Item it = load_item(kp.items, k);
    if (!(it.flags & kItemBulk)) continue;
    const SGroup& G = sgrp[it.group];
    const Scal s{G.beta1, G.omb1, G.beta2, G.omb2, G.bc1, G.bc2, G.eps, G.wd, G.lr, G.gs};
    double sq = 0.0;
    StateScale sc;
    unsigned mx[3] = {0u, 0u, 0u};
    if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB)
      sc = tensor_scales(kp, it.tensor, PASS == Pass::kScaledB);
    for (int i = bulk_vectors(it) * kVec; i < it.n; ++i) {
      if constexpr (PASS == Pass::kScan) {
        bad |= !isfinite(__fmul_rn(load1<GT>(it.g, i), s.gs));
      } else if constexpr (PASS == Pass::kNorm) {
        const double x = load1<GT>(it.g, i);
        sq += x * x;
      } else if constexpr (PASS == Pass::kReduce) {
        bad |= reduce_elem<GT>(kp, it, i, s.gs, screen);
      } else if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) {
        if (G.bits & kGroupAdamW) update_elem<true, ST, GT, OT, REM, PASS, UNIT>(it, s, i, dst, &sc, mx);
        else update_elem<false, ST, GT, OT, REM, PASS, UNIT>(it, s, i, dst, &sc, mx);
      } else {
        if (G.bits & kGroupAdamW) update_elem<true, ST, GT, OT, REM, Pass::kUpdate, UNIT>(it, s, i, dst);
        else update_elem<false, ST, GT, OT, REM, Pass::kUpdate, UNIT>(it, s, i, dst);
      }
    }
    if constexpr (PASS == Pass::kScaledA) {  // this lane's item alone: no warp reduction
      if (bulk_vectors(it) * kVec < it.n)
        for (int k = 0; k < 3; ++k) atomicMax(kp.absmax + 3 * it.tensor + k, mx[k] + 1u);
    }
    if constexpr (PASS == Pass::kNorm) {  // the item's slot, after the chunk slots
      kp.partials[kp.n_chunks + k] = static_cast<double>(G.gs) * G.gs * sq;
      __threadfence();
    }
  }
  return bad;
}

// Phase B, the rest: this CTA's items that are not 16-byte aligned, by the
// whole CTA (128-bit streaming loads when vector-aligned, then element by
// element).  Without the bulk pipeline every item goes this way.  The
// threads first test kBlock items' flags at once, so a range of bulk items
// is skipped in a few loads.
template <int ST, int GT, int OT, bool REM, Pass PASS, int UNIT = 0>
__device__ __forceinline__ bool rest_pass(const KParams& kp, const SGroup* sgrp, int item_begin,
                                          int item_end, double* red) {
  __shared__ int s_count;
  __shared__ int s_list[kBlock];
  // host-gradient launches take every item here, reading g from host memory
  const bool host_g = (kp.flags & kHostGrads) != 0;
  const Dests dst{kp.n_dests, kp.dst_delta};
  const bool screen = (kp.flags & kCheckFinite) != 0;
  bool bad = false;
  for (int base = item_begin; base < item_end; base += kBlock) {
    if (threadIdx.x == 0) s_count = 0;
    __syncthreads();
    const int k = base + threadIdx.x;
    if (k < item_end) {
      const uint16_t flags = __ldg(&kp.items[k].flags);
      if (host_g || !(FADAM_BULK && (flags & kItemBulk))) s_list[atomicAdd(&s_count, 1)] = k;
    }
    __syncthreads();
    const int count = s_count;
    for (int q = 0; q < count; ++q) {
      Item it = load_item(kp.items, s_list[q]);
      if (host_g)  // the same element offset within the tensor, in host memory
        it.g = kp.host_g[it.tensor] + (static_cast<const char*>(it.g) - kp.dev_g[it.tensor]);
      const SGroup& G = sgrp[it.group];
      const Scal s{G.beta1, G.omb1, G.beta2, G.omb2, G.bc1, G.bc2, G.eps, G.wd, G.lr, G.gs};
      if constexpr (PASS == Pass::kScan) {
        bad |= simt_scan<GT>(it, s.gs);
      } else if constexpr (PASS == Pass::kNorm) {
        double sq = 0.0;
        for (int i = threadIdx.x; i < it.n; i += kBlock) {
          const double x = load1<GT>(it.g, i);
          sq += x * x;
        }
        const double total = cta_sum(sq, red);
        if (threadIdx.x == 0) {
          kp.partials[kp.n_chunks + s_list[q]] = static_cast<double>(G.gs) * G.gs * total;
          __threadfence();
        }
      } else if constexpr (PASS == Pass::kReduce) {
        for (int i = threadIdx.x; i < it.n; i += kBlock) bad |= reduce_elem<GT>(kp, it, i, s.gs, screen);
      } else if constexpr (PASS == Pass::kScaledA || PASS == Pass::kScaledB) {
        const StateScale sc = tensor_scales(kp, it.tensor, PASS == Pass::kScaledB);
        unsigned mx[3] = {0u, 0u, 0u};
        if (G.bits & kGroupAdamW) simt_item<true, ST, GT, OT, REM, PASS, UNIT>(it, s, dst, &sc, mx);
        else simt_item<false, ST, GT, OT, REM, PASS, UNIT>(it, s, dst, &sc, mx);
        if constexpr (PASS == Pass::kScaledA) flush_absmax(kp, it.tensor, mx);
      } else {
        if (G.bits & kGroupAdamW) simt_item<true, ST, GT, OT, REM, Pass::kUpdate, UNIT>(it, s, dst);
        else simt_item<false, ST, GT, OT, REM, Pass::kUpdate, UNIT>(it, s, dst);
      }
    }
    __syncthreads();  // s_list is reused
  }
  return bad;
}

// One full pass: the bulk tiles of the shard (dynamically shared), then
// the rest of this CTA's items.
template <int ST, int GT, int OT, bool REM, Pass PASS, int NS, int UNIT = 0>
__device__ __forceinline__ void run_pass(const KParams& kp, const SGroup* sgrp, int item_begin,
                                         int item_end, unsigned* counter, unsigned* tail_counter,
                                         int n_items, unsigned char* smem, uint64_t* full,
                                         TileTag* tags, Producer& pr, double* red,
                                         unsigned& stage, bool& bad, bool& timed_out) {
  const bool bulk = FADAM_BULK && !(kp.flags & kHostGrads);
  if (bulk && kp.n_chunks > 0 && !timed_out)
    bulk_pass<ST, GT, OT, REM, PASS, NS, UNIT>(kp, sgrp, counter, smem, full, tags, pr, red, stage,
                                               bad, timed_out);
  // a shard without element-wise tails skips the tail pass, one whose items
  // all go through the tiles the rest pass: a global round trip each on
  // every CTA's path (the norm writes every bulk item's slot in its tail
  // pass, so it keeps it)
  // the element-wise paths multiply by reciprocal corrections where the
  // tiles do (the group record then holds reciprocals); the divisions by
  // corrections of 1 they keep (identities)
  constexpr int EU = UNIT & kRecipBc;
  if (bulk && (PASS == Pass::kNorm || !(kp.flags & kNoTails)))
    bad |= tail_pass<ST, GT, OT, REM, PASS, EU>(kp, sgrp, tail_counter, n_items);
  if (!bulk || !(kp.flags & kAllBulk))
    bad |= rest_pass<ST, GT, OT, REM, PASS, EU>(kp, sgrp, item_begin, item_end, red);
}

// Grid-wide barrier for a cooperative launch.  The wait is bounded: after
// kWaitLimitNs it records FADAM_ETIMEOUT in the status block and returns
// false instead of hanging.
// `extra` > 0 (diagnostic) makes the barrier wait for that many CTAs more
// than the grid has, so that every wait runs out.
__device__ __forceinline__ bool grid_barrier(KScratch* sc, unsigned extra) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = ld_acquire_u32(&sc->bar_gen);
    __threadfence();
    const unsigned arrived = atomicAdd(&sc->bar_count, 1u);
    if (arrived == gridDim.x + extra - 1) {
      atomicExch(&sc->bar_count, 0u);
      __threadfence();
      atomicAdd(&sc->bar_gen, 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (ld_acquire_u32(&sc->bar_gen) == gen) {
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicExch(&sc->status, FADAM_ETIMEOUT);
          atomicExch(&sc->launch_timeout, 1u);
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

// SCALED: the scaled 16-bit state instances (their own kernels, so the
// plain ones carry none of the two-pass code).  RECIP (16-bit state only):
// multiply by reciprocal bias corrections (FADAM_RECIP_BC) instead of
// dividing as the functor does; those are instances of their own, so that
// the default ones keep the register allocation of their own loops.
template <int ST, int GT, int OT, bool REM, bool SCALED = false, bool RECIP = false>
__global__ void FADAM_BOUNDS fadam_update_kernel(const __grid_constant__ KParams kp) {
  __shared__ SGroup sgrp[FADAM_MAX_GROUPS];
  __shared__ int s_noop;
  __shared__ __align__(8) uint64_t s_full[kMaxStages];
  __shared__ TileTag s_tags[kMaxStages];
  __shared__ Producer s_prod;  // used by thread 0 only
  __shared__ double s_red[3 * (kBlock / 32)];  // norm launches: partials per warp
  extern __shared__ __align__(128) unsigned char s_tiles[];
  constexpr int NS = pipeline_stages<ST, GT, REM, SCALED>();
  const bool capturable = (kp.flags & kCapturable) != 0;
  const int tid = threadIdx.x;

  // 1. prologue: scalars once per CTA
  if (tid == 0) {
    s_noop = kp.noop ? (__ldcg(kp.noop) == 1) : 0;  // only 1 means set
    if (FADAM_BULK) {
      for (int b = 0; b < NS; ++b) mbar_init(&s_full[b], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
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
      step = (kp.flags & kPreadvanced) ? s.step_old : step_add(s.step_old, 1);
    } else {
      s.lr = G.lr;
      s.gs = G.grad_scale;
      s.step_old = G.step;
      step = G.step;
    }
    s_group_step[tid] = step;
    // launches that only read g (norm, reduction) skip the corrections; the
    // others take them from the memo the previous launch left, or compute
    // the double pow (a few microseconds on this GPU's FP64 pipe)
    s.bc1 = 1.0f;
    s.bc2 = 1.0f;
    if ((G.bits & kGroupBiasCorr) && !(kp.flags & (kNormOnly | kReduceOnly)) &&
        !(kp.memo && memo_lookup(kp.memo, tid, G.beta1, G.beta2, step, s.bc1, s.bc2))) {
      s.bc1 = bias_correction(G.beta1, step);
      s.bc2 = bias_correction(G.beta2, step);
    }
    if constexpr (RECIP) {
      // the reciprocal instances keep 1/bc1 and 1/bc2 in their place (IEEE
      // reciprocals; 1 stays 1, so the launch-wide test for corrections of
      // 1 below reads the same)
      s.bc1 = __frcp_rn(s.bc1);
      s.bc2 = __frcp_rn(s.bc2);
    }
    sgrp[tid] = s;
  }
  __syncthreads();
  // the next step's corrections, for the next launch: one warp of the last
  // CTA pays the pow while the other CTAs start on the shard's tiles
  if (kp.memo && blockIdx.x == gridDim.x - 1 && !(kp.flags & (kNormOnly | kReduceOnly)) &&
      tid >= 32 && tid < 32 + kp.n_groups) {
    const SGroup& g = sgrp[tid - 32];
    if (g.bits & kGroupBiasCorr)
      memo_store(kp.memo, tid - 32, g.beta1, g.beta2, step_add(s_group_step[tid - 32], 1));
  }

  const int item_begin = __ldg(kp.cta_begin + blockIdx.x);
  const int item_end = __ldg(kp.cta_begin + blockIdx.x + 1);
  const int n_items = __ldg(kp.cta_begin + gridDim.x);
  unsigned stage = 0;  // tiles through the pipeline so far (buffer and parity)
  bool barrier_ok = true, timed_out = false;

  const bool norm_only = (kp.flags & kNormOnly) != 0;
  if (norm_only) {
    // squared gradient norm instead of the update: one weighted partial per
    // chunk of tiles and per item (tails, unaligned items), summed by the
    // last CTA below in a fixed order
    bool unused = false;
    run_pass<ST, GT, OT, REM, Pass::kNorm, NS>(kp, sgrp, item_begin, item_end, &kp.scratch->next_scan,
                                           &kp.scratch->next_tail_scan, n_items, s_tiles, s_full,
                                           s_tags, s_prod, s_red, stage, unused, timed_out);
  }

  // 1b. the reduce-scatter stand-in: this rank's g from the exchange
  //     sources (alone, or before the update; it runs even when the step
  //     is then skipped), screened in the same pass when the plan asks
  const bool reduce_only = (kp.flags & kReduceOnly) != 0;
  const bool reduce_first = (kp.flags & kReduceFirst) != 0;
  const bool updates = !norm_only && !reduce_only;
  if (reduce_only || reduce_first) {
    bool bad = false;
    run_pass<ST, GT, OT, REM, Pass::kReduce, NS>(kp, sgrp, item_begin, item_end, &kp.scratch->next_scan,
                                             &kp.scratch->next_tail_scan, n_items, s_tiles, s_full,
                                             s_tags, s_prod, s_red, stage, bad, timed_out);
    // the update copies g with the async proxy: order this thread's
    // generic-proxy stores of g before that
    asm volatile("fence.proxy.async.global;" ::: "memory");
    if (reduce_first) {
      // warp-level OR of the screen: one write of the flag per warp that saw
      // a value that is not finite (the grid barrier orders it before the
      // flag is read)
      if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) atomicExch(kp.noop, 1);
      barrier_ok = grid_barrier(kp.scratch, (kp.flags & kTestBarrierTimeout) ? 1u : 0u);
      if (tid == 0) {
        s_noop = kp.noop ? (ld_acquire_s32(kp.noop) == 1) : 0;
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncthreads();
    }
  }

  // 2. optional inf/nan screen over the whole shard before any update
  if (updates && !reduce_first && (kp.flags & kCheckFinite)) {
    bool bad = false;
    if (!s_noop)
      run_pass<ST, GT, OT, REM, Pass::kScan, NS>(kp, sgrp, item_begin, item_end, &kp.scratch->next_scan,
                                         &kp.scratch->next_tail_scan, n_items, s_tiles, s_full,
                                         s_tags, s_prod, s_red, stage, bad, timed_out);
    // warp-level OR of the screen, one write of the flag per warp that saw
    // a value that is not finite; the grid barrier orders the writes before
    // every CTA reads the flag
    if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) atomicExch(kp.noop, 1);
    barrier_ok = grid_barrier(kp.scratch, (kp.flags & kTestBarrierTimeout) ? 1u : 0u);
    if (tid == 0) s_noop = (ld_acquire_s32(kp.noop) == 1);
    __syncthreads();
  }

  // 3. the update (scaled 16-bit state: the absmax pass, a bounded grid
  //    barrier, the rescale pass)
  bool scaled_done = false;
  if (updates && !s_noop && barrier_ok) {
    // bias corrections that are 1 in every group: the same for every CTA
    int unit = 0;
    if constexpr (unit_bc_instances<ST, REM>()) {
      unit = kUnitBc1 | kUnitBc2;
      for (int k = 0; k < kp.n_groups; ++k) {
        if (sgrp[k].bc1 != 1.0f) unit &= ~kUnitBc1;
        if (sgrp[k].bc2 != 1.0f) unit &= ~kUnitBc2;
      }
    }
    bool unused = false;
    // the update passes for a compile-time unit mask U
    auto passes = [&](auto unit_c) {
      constexpr int U = decltype(unit_c)::value;
      if constexpr (SCALED) {
        run_pass<ST, GT, OT, REM, Pass::kScaledA, NS, U>(kp, sgrp, item_begin, item_end,
                                                         &kp.scratch->next_update,
                                                         &kp.scratch->next_tail_update, n_items,
                                                         s_tiles, s_full, s_tags, s_prod, s_red,
                                                         stage, unused, timed_out);
        // the timeout diagnostic of a plan without the screen acts here
        barrier_ok = grid_barrier(
            kp.scratch, ((kp.flags & kTestBarrierTimeout) && !(kp.flags & kCheckFinite)) ? 1u : 0u);
        if (barrier_ok)
          run_pass<ST, GT, OT, REM, Pass::kScaledB, NS, U>(kp, sgrp, item_begin, item_end,
                                                           &kp.scratch->next_rescale,
                                                           &kp.scratch->next_tail_rescale, n_items,
                                                           s_tiles, s_full, s_tags, s_prod, s_red,
                                                           stage, unused, timed_out);
        scaled_done = barrier_ok;
      } else {
        run_pass<ST, GT, OT, REM, Pass::kUpdate, NS, U>(kp, sgrp, item_begin, item_end,
                                                        &kp.scratch->next_update,
                                                        &kp.scratch->next_tail_update, n_items,
                                                        s_tiles, s_full, s_tags, s_prod, s_red,
                                                        stage, unused, timed_out);
      }
    };
    if constexpr (unit_bc_instances<ST, REM>() && RECIP) {
      // reciprocals: one loop for any correction that is not 1 (the product
      // by a reciprocal of 1 is exact), one for both corrections at 1
      if (unit == (kUnitBc1 | kUnitBc2)) passes(std::integral_constant<int, kUnitBc1 | kUnitBc2>{});
      else passes(std::integral_constant<int, kRecipBc>{});
    } else if constexpr (unit_bc_instances<ST, REM>()) {
      if (unit == (kUnitBc1 | kUnitBc2)) passes(std::integral_constant<int, kUnitBc1 | kUnitBc2>{});
      else if (unit == kUnitBc1) passes(std::integral_constant<int, kUnitBc1>{});
      else passes(std::integral_constant<int, 0>{});
    } else {
      passes(std::integral_constant<int, 0>{});
    }
  }
  if (__syncthreads_or(timed_out) && tid == 0) {
    atomicExch(&kp.scratch->status, FADAM_ETIMEOUT);
    atomicExch(&kp.scratch->launch_timeout, 1u);
  }

  // 4. the last CTA to finish resets the work counters for the next launch
  //    and, for capturable plans, advances the step counters; for a norm
  //    launch it sums the partials
  __shared__ int s_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&kp.scratch->done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (norm_only && s_last) {
    __threadfence();
    const int n_slots = (FADAM_BULK ? kp.n_chunks : 0) + n_items;
    const int base = FADAM_BULK ? 0 : kp.n_chunks;
    double x = 0.0;
    for (int i = tid; i < n_slots; i += kBlock) x += __ldcg(kp.partials + base + i);
    const double total = cta_sum(x, s_red);
    if (tid == 0) *kp.sumsq_out = total;
  }
  if (SCALED && updates && s_last) {
    // the new scales replace the old (tensors that had no element keep
    // theirs), unless some wait of this launch gave up; the absmax slots
    // are cleared for the next step either way, also when this CTA's own
    // wait between the passes gave up (other CTAs may have filled them)
    __threadfence();
    const bool ok = scaled_done && ld_acquire_u32(&kp.scratch->launch_timeout) == 0u;
    for (int j = tid; j < 3 * kp.n_tensors; j += kBlock) {
      const unsigned a = __ldcg(kp.absmax + j);
      if (a) {
        if (ok) kp.scales[j] = __fdiv_rn(__uint_as_float(a - 1u), kp.max_scaled);
        kp.absmax[j] = 0u;
      }
    }
  }
  // every thread of the last CTA has read this launch's timeout flag before
  // thread 0 clears it below
  __syncthreads();
  if (tid == 0) {
    if (s_last) {
      __threadfence();
      if (updates && capturable && !(kp.flags & kPreadvanced)) {
        const int adv = (s_noop || !barrier_ok) ? 0 : 1;
        for (int g = 0; g < kp.n_groups; ++g)
          if (sgrp[g].bits & kGroupOwnsStep)
            *kp.groups[g].step_dev = step_add(sgrp[g].step_old, adv);
      }
      atomicExch(&kp.scratch->next_update, 0u);
      atomicExch(&kp.scratch->next_scan, 0u);
      atomicExch(&kp.scratch->next_tail_update, 0u);
      atomicExch(&kp.scratch->next_tail_scan, 0u);
      atomicExch(&kp.scratch->next_rescale, 0u);
      atomicExch(&kp.scratch->next_tail_rescale, 0u);
      // every CTA has left its grid barriers by now: a wait that gave up
      // leaves its arrival counted, which would stall the next launch's
      // barrier, so the count starts from zero again (the status word keeps
      // the timeout until fadam_plan_status reads it)
      atomicExch(&kp.scratch->bar_count, 0u);
      atomicExch(&kp.scratch->launch_timeout, 0u);
      atomicExch(&kp.scratch->done, 0u);
    }
  }
}

// Entry for one (state dtype, g dtype): every out dtype, and the remainder
// form (bf16 high half + int16 remainder, fp32 m and v) under fp32 state.
template <int ST, int GT>
KernelEntry kernel_for(int out_dtype, bool remainders) {
  if (remainders) {
    // only the fp32 state form has a remainder instance
    if constexpr (ST == FADAM_DT_F32) {
      if (out_dtype != FADAM_DT_BF16) return {nullptr, 0};
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_BF16, true>),
              smem_bytes<ST, GT, true>()};
    } else {
      return {nullptr, 0};
    }
  }
  const size_t smem = smem_bytes<ST, GT, false>();
  switch (out_dtype) {
    case FADAM_DT_NONE:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_NONE, false>), smem};
    case FADAM_DT_F32:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F32, false>), smem};
    case FADAM_DT_BF16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_BF16, false>), smem};
    case FADAM_DT_F16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F16, false>), smem};
    default: return {nullptr, 0};
  }
}

// The scaled 16-bit state instance for a (state dtype, g dtype, out dtype)
// combination; the state dtype is bf16 or fp16.
template <int ST, int GT>
KernelEntry scaled_kernel_for(int out_dtype) {
  const size_t smem = smem_bytes<ST, GT, false, true>();
  switch (out_dtype) {
    case FADAM_DT_NONE:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_NONE, false, true>), smem};
    case FADAM_DT_F32:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F32, false, true>), smem};
    case FADAM_DT_BF16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_BF16, false, true>), smem};
    case FADAM_DT_F16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F16, false, true>), smem};
    default: return {nullptr, 0};
  }
}

// The instances with reciprocal bias corrections (FADAM_RECIP_BC) of a
// 16-bit state dtype (ST bf16 or fp16), plain or scaled: every out dtype.
template <int ST, int GT, bool SCALED>
KernelEntry recip_kernel_for(int out_dtype) {
  const size_t smem = smem_bytes<ST, GT, false, SCALED>();
  switch (out_dtype) {
    case FADAM_DT_NONE:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_NONE, false, SCALED, true>), smem};
    case FADAM_DT_F32:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F32, false, SCALED, true>), smem};
    case FADAM_DT_BF16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_BF16, false, SCALED, true>), smem};
    case FADAM_DT_F16:
      return {reinterpret_cast<const void*>(&fadam_update_kernel<ST, GT, FADAM_DT_F16, false, SCALED, true>), smem};
    default: return {nullptr, 0};
  }
}

}  // namespace fadam
