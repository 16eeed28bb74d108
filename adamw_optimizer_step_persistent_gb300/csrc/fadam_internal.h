// Internal layout shared by the host planner (fadam_plan.cu) and the kernel
// translation units (fadam_kernels_g*.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fadam.h"

namespace fadam {

// Threads per CTA of the update kernel.
#ifndef FADAM_BLOCK
#define FADAM_BLOCK 1024
#endif
constexpr int kBlock = FADAM_BLOCK;
static_assert(kBlock % 32 == 0 && kBlock >= 32 && kBlock <= 1024,
              "threads per CTA: whole warps, at most 1024");
// State forms of the kernel's ST template argument: FADAM_DT_F32, _BF16 or
// _F16 mean p, m and v all of that dtype; these two mean an fp32 master with
// m and v in bf16 or fp16 (exp_avg_dtype = exp_avg_sq_dtype).
constexpr int kStateF32MomBF16 = 4;
constexpr int kStateF32MomF16 = 5;
__host__ __device__ constexpr int p_dtype_of(int st) {
  return st == kStateF32MomBF16 || st == kStateF32MomF16 ? FADAM_DT_F32 : st;
}
__host__ __device__ constexpr int mv_dtype_of(int st) {
  return st == kStateF32MomBF16 ? FADAM_DT_BF16 : st == kStateF32MomF16 ? FADAM_DT_F16 : st;
}

// Elements per vector access (one 16-byte fp32 vector).
constexpr int kVec = 4;
// Largest work item, in elements (keeps in-item indices in 32 bits).
constexpr int64_t kMaxItem = int64_t(1) << 26;
// Work items are cut at multiples of this many elements.
constexpr int64_t kCutQuantum = 32;

// Tiles of the bulk pipeline: kBlock 4-element vectors each (one per
// thread); a chunk, the unit CTAs pull from the shared work counter, is at
// most kChunkTiles tiles of one item.
constexpr int kChunkTiles = 16;

// Item flags.
constexpr uint16_t kItemVec = 1;   // every stream is aligned to one 4-element vector
constexpr uint16_t kItemBulk = 2;  // ... and to 16 bytes (bulk copies allowed)

// One contiguous run of one tensor: pointers already offset to the run start.
struct alignas(16) Item {
  void* p;
  void* m;
  void* v;
  const void* g;
  void* p_out;
  int16_t* rem;
  int32_t n;        // elements in the run
  uint16_t group;   // param group
  uint16_t flags;   // kItemVec, kItemBulk
  int32_t tensor;   // index of the tensor the run belongs to
};
static_assert(sizeof(Item) == 64, "Item is one 64-byte record");

// Group bits.
constexpr uint32_t kGroupAdamW = 1;      // decoupled weight decay
constexpr uint32_t kGroupBiasCorr = 2;   // bias correction on
constexpr uint32_t kGroupOwnsStep = 4;   // advances *step_dev (first user of the pointer)

// One param group as the kernel sees it (passed by value).
struct alignas(16) KGroup {
  float beta1, beta2, eps, wd;
  float lr, grad_scale;   // regular plans
  int32_t step;           // regular plans: the step of this update
  uint32_t bits;          // kGroup*
  const float* lr_dev;    // capturable plans
  const float* gs_dev;
  int32_t* step_dev;
  int64_t reserved;
};
static_assert(sizeof(KGroup) == 64, "KGroup is one 64-byte record");

// Bias corrections of one group for one step, kept between launches.  The
// double-precision pow behind them takes microseconds on this GPU's narrow
// FP64 pipe, on the path of every CTA; instead one CTA of each launch
// computes the next step's corrections and the next launch reads them.  It
// is a memo of a pure function of (beta1, beta2, step): an entry serves only
// when all three match and its tag is set, else the launch computes the
// corrections itself.  Two entries per group, chosen by the step's parity,
// so that a launch never writes an entry its own CTAs read.
struct alignas(16) BcMemo {
  uint32_t beta1_bits, beta2_bits;
  int32_t step;
  uint32_t tag;  // kMemoTag once written
  float bc1, bc2;
  int32_t reserved[2];
};
static_assert(sizeof(BcMemo) == 32, "BcMemo is two 16-byte words");
constexpr uint32_t kMemoTag = 0x62634d4du;
constexpr int kMemoEntries = 2 * FADAM_MAX_GROUPS;

// Per-plan device status block.
// One chunk of bulk tiles: tiles [tile0, tile0 + ntiles) of item `item`.
struct alignas(16) Chunk {
  int32_t item;
  int32_t tile0;
  int32_t ntiles;
  int32_t reserved;
};

struct KScratch {
  unsigned int done;         // CTAs finished in the current launch (last one resets all)
  unsigned int bar_count;    // grid barrier arrivals
  unsigned int bar_gen;      // grid barrier generation
  int status;                // FADAM_OK or FADAM_ETIMEOUT
  unsigned int next_update;  // next chunk of the update's bulk pass
  unsigned int next_scan;    // next chunk of the inf/nan screen's bulk pass
  unsigned int next_tail_update;  // next item whose tail the update takes
  unsigned int next_tail_scan;    // next item whose tail the screen takes
  unsigned int next_rescale;      // scaled state: next chunk of the rescale pass
  unsigned int next_tail_rescale; // ... and next item whose tail it takes
  unsigned int launch_timeout;    // 1 once a wait of the current launch gave up
                                  // (status keeps it until read; this one is
                                  // cleared by the launch's last CTA)
};

// Kernel flags.
constexpr uint32_t kCapturable = FADAM_CAPTURABLE;
constexpr uint32_t kCheckFinite = FADAM_CHECK_FINITE;
constexpr uint32_t kPreadvanced = FADAM_STEP_PREADVANCED;
constexpr uint32_t kTestBarrierTimeout = FADAM_TEST_BARRIER_TIMEOUT;
constexpr uint32_t kScaledStates = FADAM_SCALED_STATES;
// Launch-only flags (never plan flags): compute the squared gradient norm
// instead of the update; write the gradient shard from the exchange sources
// (alone, or before the update with a grid barrier between).
constexpr uint32_t kNormOnly = 1u << 30;
constexpr uint32_t kReduceOnly = 1u << 29;
constexpr uint32_t kReduceFirst = 1u << 28;
// Launch-only: the gradients are read from pinned host memory (zero copy):
// tensor t's g lives at host_g[t] instead of dev_g[t], every item goes the
// element-wise way (plain loads; no bulk copies from host memory).
constexpr uint32_t kHostGrads = 1u << 27;
// Launch-only, from the plan's shape: no bulk item has an element-wise tail
// (every bulk item's length is a multiple of 8), and no item is off the
// bulk path.  They let a launch skip the tail and rest passes.
constexpr uint32_t kNoTails = 1u << 26;
constexpr uint32_t kAllBulk = 1u << 25;

// The exchange's reduction: divide the sum by R (ReduceOp.AVG); add the
// reduced value to the shard's old g (gradient accumulation).
constexpr int32_t kExchangeAverage = FADAM_EXCHANGE_AVERAGE;
constexpr int32_t kExchangeAccumulate = FADAM_EXCHANGE_ACCUMULATE;

// Everything one launch needs, passed as a __grid_constant__ parameter.
struct alignas(16) KParams {
  const Item* items;
  const int32_t* cta_begin;  // grid+1 entries: CTA b runs items [cta_begin[b], cta_begin[b+1])
  int32_t* noop;             // may be null
  KScratch* scratch;
  const Chunk* chunks;       // bulk tiles, pulled dynamically by the CTAs
  double* partials;          // norm launches: weighted sums of squares, one per chunk then one per item
  double* sumsq_out;         // norm launches: sum_g grad_scale_g^2 * sum g^2
  BcMemo* memo;              // kMemoEntries bias-correction entries, or null
  int32_t n_chunks;
  int32_t n_groups;
  uint32_t flags;
  int32_t reserved;
  // the data-parallel exchange: byte offsets from the shard's g to each
  // source's, and from p_out to each extra destination
  int32_t n_sources;
  int32_t average;  // kExchangeAverage | kExchangeAccumulate
  int32_t n_dests;
  float avg_mul;  // 1/R when averaging over a power-of-two R (exact), else 0
  int64_t src_delta[FADAM_MAX_SOURCES];
  int64_t dst_delta[FADAM_MAX_DESTS];
  // scaled state: 3 scales per tensor (p, m, v), the new-value absmax of
  // each (1 + largest |x| bit pattern; 0 = no element seen), and the scale
  // target (half the state dtype's largest finite value)
  float* scales;
  unsigned* absmax;
  int32_t n_tensors;
  float max_scaled;
  // host-gradient launches: per tensor, the device-accessible address of
  // the host gradient and the tensor's own device g
  const char* const* host_g;
  const char* const* dev_g;
  KGroup groups[FADAM_MAX_GROUPS];
};

// A kernel and the dynamic shared memory (bulk-copy tiles) it launches with.
struct KernelEntry {
  const void* fn;
  size_t smem;
};

// Kernel entry for the (state dtype, g dtype, out dtype, remainders)
// combination, or a null fn when the combination does not exist.  One
// function per (state, g) pair, each in fadam_kernels_s<state>_g<g>.cu.
#define FADAM_DECLARE_KERNELS(S, G) KernelEntry kernel_s##S##_g##G(int out_dtype, bool remainders);
FADAM_DECLARE_KERNELS(f32, f32)
FADAM_DECLARE_KERNELS(f32, bf16)
FADAM_DECLARE_KERNELS(f32, f16)
FADAM_DECLARE_KERNELS(bf16, f32)
FADAM_DECLARE_KERNELS(bf16, bf16)
FADAM_DECLARE_KERNELS(bf16, f16)
FADAM_DECLARE_KERNELS(f16, f32)
FADAM_DECLARE_KERNELS(f16, bf16)
FADAM_DECLARE_KERNELS(f16, f16)
FADAM_DECLARE_KERNELS(f32mbf16, f32)
FADAM_DECLARE_KERNELS(f32mbf16, bf16)
FADAM_DECLARE_KERNELS(f32mbf16, f16)
FADAM_DECLARE_KERNELS(f32mf16, f32)
FADAM_DECLARE_KERNELS(f32mf16, bf16)
FADAM_DECLARE_KERNELS(f32mf16, f16)
#undef FADAM_DECLARE_KERNELS

// Scaled 16-bit state instances (state dtype bf16 or fp16), one function per
// (state, g) pair, each in fadam_kernels_scaled_s<state>_g<g>.cu.
#define FADAM_DECLARE_SCALED(S, G) KernelEntry scaled_kernel_s##S##_g##G(int out_dtype);
FADAM_DECLARE_SCALED(bf16, f32)
FADAM_DECLARE_SCALED(bf16, bf16)
FADAM_DECLARE_SCALED(bf16, f16)
FADAM_DECLARE_SCALED(f16, f32)
FADAM_DECLARE_SCALED(f16, bf16)
FADAM_DECLARE_SCALED(f16, f16)
#undef FADAM_DECLARE_SCALED

// Instances of the 16-bit state forms with reciprocal bias corrections
// (FADAM_RECIP_BC), plain and scaled, one function per (state, g) pair, in
// fadam_kernels_recip_s<state>_g<g>.cu and fadam_kernels_recip_scaled_*.cu.
#define FADAM_DECLARE_RECIP(S, G)                       \
  KernelEntry recip_kernel_s##S##_g##G(int out_dtype);  \
  KernelEntry recip_scaled_kernel_s##S##_g##G(int out_dtype);
FADAM_DECLARE_RECIP(bf16, f32)
FADAM_DECLARE_RECIP(bf16, bf16)
FADAM_DECLARE_RECIP(bf16, f16)
FADAM_DECLARE_RECIP(f16, f32)
FADAM_DECLARE_RECIP(f16, bf16)
FADAM_DECLARE_RECIP(f16, f16)
#undef FADAM_DECLARE_RECIP

}  // namespace fadam
