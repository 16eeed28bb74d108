// Host side of the C ABI: argument checks, the tensor-list packer that
// builds the persistent grid's balanced work list, plan lifecycle and the
// launches.  Every check runs before the first CUDA call, so a rejected call
// launches nothing.
//
// The packer replaces the fixed-size chunk table of the page's
// multi_tensor_apply (one CTA per chunk, several launches when the table is
// full; "Enhance Distributed Fused Adam (#1794)", operator() reading
// block_to_tensor / block_to_chunk) with one launch whose CTAs each take a
// contiguous, equal-cost slice of the concatenated shard.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "fadam.h"
#include "fadam_internal.h"

using namespace fadam;

namespace {

// Bytes of work that justify one more CTA for small shards.
constexpr double kMinCtaCost = 64.0 * 1024.0;
// Fixed cost of one work item, in byte-equivalents (descriptor fetch, tail).
constexpr double kItemOverhead = 4096.0;
// Most chunks a plan's work list holds (chunks grow past kChunkTiles tiles
// beyond that).
constexpr int64_t kPlanMaxChunks = 131072;
// Smallest chunk of the tapered end of a chunk list, in tiles.
#ifndef FADAM_TAPER_MIN_TILES
#define FADAM_TAPER_MIN_TILES 4
#endif
constexpr int64_t kTaperMinTiles = FADAM_TAPER_MIN_TILES;
// Largest tensor the library accepts, in elements.
constexpr int64_t kMaxNumel = int64_t(1) << 40;

thread_local std::string t_last_error;

fadam_status fail(fadam_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

fadam_status cuda_fail(cudaError_t e, const char* what) {
  t_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  (void)cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return FADAM_ECUDA;
}

int elem_size(int32_t dt) {
  switch (dt) {
    case FADAM_DT_F32: return 4;
    case FADAM_DT_BF16:
    case FADAM_DT_F16: return 2;
    default: return 0;
  }
}

bool finite(float x) { return std::isfinite(x); }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  int want;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) : want(dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != want) err = cudaSetDevice(want);
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != want) cudaSetDevice(prev);
  }
};

struct Dtypes {
  int32_t p, g, out;  // p: the state dtype of p, m, v (bf16 high half in remainder form)
  bool rem;
  int32_t mv = FADAM_DT_NONE;  // 16-bit moments under an fp32 master (FADAM_MOMENTS_*)
};

Dtypes make_dtypes(int32_t p, int32_t g, int32_t out, uint32_t flags) {
  Dtypes d{p, g, out, (flags & FADAM_REMAINDERS) != 0};
  if (flags & FADAM_MOMENTS_BF16) d.mv = FADAM_DT_BF16;
  if (flags & FADAM_MOMENTS_F16) d.mv = FADAM_DT_F16;
  return d;
}

// Element size of m and v: the state dtype, the moments' own dtype, or fp32
// in the remainder form.
int mv_size(const Dtypes& d) {
  return d.rem ? 4 : elem_size(d.mv != FADAM_DT_NONE ? d.mv : d.p);
}

fadam_status check_dtypes(const Dtypes& d, uint32_t flags) {
  const uint32_t known = FADAM_CAPTURABLE | FADAM_REMAINDERS | FADAM_CHECK_FINITE |
                         FADAM_STEP_PREADVANCED | FADAM_TEST_BARRIER_TIMEOUT |
                         FADAM_SCALED_STATES | FADAM_MOMENTS_BF16 | FADAM_MOMENTS_F16 |
                         FADAM_RECIP_BC;
  if (flags & ~known) return fail(FADAM_EINVAL, "unknown flag bits 0x%x", flags & ~known);
  if ((flags & FADAM_MOMENTS_BF16) && (flags & FADAM_MOMENTS_F16))
    return fail(FADAM_EINVAL, "FADAM_MOMENTS_BF16 and FADAM_MOMENTS_F16 exclude each other");
  if (d.mv != FADAM_DT_NONE &&
      (d.p != FADAM_DT_F32 || d.rem || (flags & FADAM_SCALED_STATES)))
    return fail(FADAM_EDTYPE, "16-bit moments need an fp32 master (no remainders, no scaled "
                              "states)");
  if ((flags & FADAM_STEP_PREADVANCED) && !(flags & FADAM_CAPTURABLE))
    return fail(FADAM_EINVAL, "FADAM_STEP_PREADVANCED needs FADAM_CAPTURABLE");
  if ((flags & FADAM_TEST_BARRIER_TIMEOUT) && !(flags & (FADAM_CHECK_FINITE | FADAM_SCALED_STATES)))
    return fail(FADAM_EINVAL, "FADAM_TEST_BARRIER_TIMEOUT needs FADAM_CHECK_FINITE or "
                              "FADAM_SCALED_STATES (a grid barrier to run out)");
  if (d.g != FADAM_DT_F32 && d.g != FADAM_DT_BF16 && d.g != FADAM_DT_F16)
    return fail(FADAM_EDTYPE, "g dtype %d is not fp32, bf16 or fp16", d.g);
  if (d.out != FADAM_DT_NONE && elem_size(d.out) == 0)
    return fail(FADAM_EDTYPE, "param-out dtype %d is not none, fp32, bf16 or fp16", d.out);
  if (d.rem) {
    if (d.p != FADAM_DT_BF16)
      return fail(FADAM_EDTYPE, "remainder mode needs bf16 params (p dtype %d)", d.p);
    if (d.out != FADAM_DT_BF16)
      return fail(FADAM_EDTYPE, "remainder mode writes a bf16 param-out (out dtype %d)", d.out);
  } else if (elem_size(d.p) == 0) {
    return fail(FADAM_EDTYPE, "state dtype %d (p, m, v) is not fp32, bf16 or fp16", d.p);
  }
  if ((flags & FADAM_SCALED_STATES) && (d.rem || (d.p != FADAM_DT_BF16 && d.p != FADAM_DT_F16)))
    return fail(FADAM_EDTYPE, "scaled states need a bf16 or fp16 state and no remainders");
  return FADAM_OK;
}

fadam_status check_groups(const fadam_group* groups, int32_t n_groups, uint32_t flags,
                          const std::vector<char>& has_tensor, bool check_host_step) {
  if (n_groups < 1 || n_groups > FADAM_MAX_GROUPS)
    return fail(FADAM_EINVAL, "n_groups %d outside 1..%d", n_groups, FADAM_MAX_GROUPS);
  if (!groups) return fail(FADAM_EINVAL, "groups is NULL");
  const bool capt = flags & FADAM_CAPTURABLE;
  for (int32_t i = 0; i < n_groups; ++i) {
    const fadam_group& g = groups[i];
    if (g.mode != FADAM_MODE_L2 && g.mode != FADAM_MODE_ADAMW)
      return fail(FADAM_EINVAL, "group %d: mode %d is neither L2 (0) nor AdamW (1)", i, g.mode);
    if (g.bias_correction != 0 && g.bias_correction != 1)
      return fail(FADAM_EINVAL, "group %d: bias_correction %d is not 0 or 1", i, g.bias_correction);
    if (!(g.beta1 >= 0.0f && g.beta1 < 1.0f) || !(g.beta2 >= 0.0f && g.beta2 < 1.0f))
      return fail(FADAM_EINVAL, "group %d: betas (%g, %g) outside [0, 1)", i, g.beta1, g.beta2);
    if (!(g.eps >= 0.0f) || !finite(g.eps))
      return fail(FADAM_EINVAL, "group %d: eps %g is not finite and >= 0", i, g.eps);
    if (!finite(g.weight_decay))
      return fail(FADAM_EINVAL, "group %d: weight_decay is not finite", i);
    if (capt) {
      if (!g.step_dev) return fail(FADAM_EINVAL, "group %d: capturable plan without step_dev", i);
      if (reinterpret_cast<uintptr_t>(g.step_dev) % 4)
        return fail(FADAM_EALIGN, "group %d: step_dev is not 4-byte aligned", i);
      if (has_tensor[i] && (!g.lr_dev || !g.grad_scale_dev))
        return fail(FADAM_EINVAL, "group %d: capturable plan needs lr_dev and grad_scale_dev", i);
      if ((g.lr_dev && reinterpret_cast<uintptr_t>(g.lr_dev) % 4) ||
          (g.grad_scale_dev && reinterpret_cast<uintptr_t>(g.grad_scale_dev) % 4))
        return fail(FADAM_EALIGN, "group %d: lr_dev / grad_scale_dev not 4-byte aligned", i);
    } else {
      if (!finite(g.lr) || !finite(g.grad_scale))
        return fail(FADAM_EINVAL, "group %d: lr or grad_scale is not finite", i);
      if (check_host_step && g.bias_correction == 1 && g.step < 1)
        return fail(FADAM_EINVAL, "group %d: step %d < 1 with bias correction (1-beta^step = 0)",
                    i, g.step);
    }
  }
  return FADAM_OK;
}

bool misaligned(const void* ptr, int esz) {
  return reinterpret_cast<uintptr_t>(ptr) % static_cast<uintptr_t>(esz) != 0;
}

fadam_status check_tensors(const fadam_tensor* ts, int64_t n, int32_t n_groups, const Dtypes& d,
                           std::vector<char>& has_tensor) {
  if (n < 0) return fail(FADAM_EINVAL, "n_tensors %lld < 0", (long long)n);
  if (n > 0 && !ts) return fail(FADAM_EINVAL, "tensors is NULL");
  if (n > (int64_t(1) << 31)) return fail(FADAM_ELIMIT, "n_tensors %lld > 2^31", (long long)n);
  const int psz = elem_size(d.p), gsz = elem_size(d.g), osz = elem_size(d.out);
  for (int64_t i = 0; i < n; ++i) {
    const fadam_tensor& t = ts[i];
    if (t.group < 0 || t.group >= n_groups)
      return fail(FADAM_EINVAL, "tensor %lld: group %d outside 0..%d", (long long)i, t.group,
                  n_groups - 1);
    if (t.numel < 0) return fail(FADAM_EINVAL, "tensor %lld: numel < 0", (long long)i);
    if (t.numel > kMaxNumel)
      return fail(FADAM_ELIMIT, "tensor %lld: numel %lld > 2^40", (long long)i, (long long)t.numel);
    if (t.numel == 0) continue;
    has_tensor[t.group] = 1;
    if (!t.p || !t.m || !t.v || !t.g)
      return fail(FADAM_EINVAL, "tensor %lld: p, m, v and g must be non-NULL", (long long)i);
    if (d.out == FADAM_DT_NONE ? t.p_out != nullptr : t.p_out == nullptr)
      return fail(FADAM_EINVAL, "tensor %lld: p_out must be %s for param-out dtype %d",
                  (long long)i, d.out == FADAM_DT_NONE ? "NULL" : "non-NULL", d.out);
    if (d.rem ? t.rem == nullptr : t.rem != nullptr)
      return fail(FADAM_EINVAL, "tensor %lld: rem must be %s", (long long)i,
                  d.rem ? "non-NULL in remainder mode" : "NULL outside remainder mode");
    if (misaligned(t.p, psz) || misaligned(t.m, mv_size(d)) || misaligned(t.v, mv_size(d)) ||
        misaligned(t.g, gsz) ||
        (t.p_out && misaligned(t.p_out, osz)) || (t.rem && misaligned(t.rem, 2)))
      return fail(FADAM_EALIGN, "tensor %lld: a pointer is not aligned to its element size",
                  (long long)i);
  }
  return FADAM_OK;
}

// Algorithmic bytes per element: every stream read or written once.
double bytes_per_elem(const Dtypes& d) {
  const int gsz = elem_size(d.g);
  if (d.rem) return 2 + 2 + 2 + 2 + 8 + 8 + gsz;  // p_hi R, p_out W, rem R+W, m, v, g
  // p, m, v read and written, g read, p_out written
  return 2.0 * elem_size(d.p) + 4.0 * mv_size(d) + gsz + elem_size(d.out);
}

struct PackItem {
  int64_t tensor;
  int64_t offset;
  int64_t n;
  int level;  // 0 scalar, 1 vector-aligned, 2 also 16-byte aligned
};

struct Piece {
  int64_t tensor, offset, n;
  int level;
};

struct Head {
  int64_t h;  // elements to peel off the start of the tensor
  int level;  // alignment of the rest, as in PackItem
};

// How many leading elements to peel so that the rest of the tensor is as
// aligned as possible: every stream 16-byte aligned (bulk copies), else
// every stream aligned to one 4-element vector, else nothing (scalar path).
Head body_alignment(const fadam_tensor& t, const Dtypes& d) {
  const void* ptrs[6] = {t.p, t.m, t.v, t.g, t.p_out, t.rem};
  const int esz[6] = {elem_size(d.p), mv_size(d), mv_size(d), elem_size(d.g), elem_size(d.out), 2};
  for (int64_t h = 0; h < 8; ++h) {
    bool ok = true;
    for (int s = 0; s < 6 && ok; ++s)
      if (ptrs[s] && esz[s] && (reinterpret_cast<uintptr_t>(ptrs[s]) + h * esz[s]) % 16 != 0) ok = false;
    if (ok) return {h, 2};
  }
  int64_t r = -1;
  for (int s = 0; s < 6; ++s) {
    if (!ptrs[s] || esz[s] == 0) continue;
    const int64_t rs = static_cast<int64_t>((reinterpret_cast<uintptr_t>(ptrs[s]) / esz[s]) % kVec);
    if (r < 0) r = rs;
    else if (r != rs) return {0, 0};
  }
  return {r < 0 ? 0 : (kVec - r) % kVec, 1};
}

// Split the shard into pieces (aligned bodies, scalar heads) and cut them
// into items so that CTA b's items cost about total/grid each.
void pack(const fadam_tensor* ts, int64_t n, const Dtypes& d, int grid,
          std::vector<PackItem>& items, std::vector<int32_t>& cta_begin) {
  std::vector<Piece> pieces;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t len = ts[i].numel;
    if (len <= 0) continue;
    const Head hd = body_alignment(ts[i], d);
    if (hd.level == 0) {
      pieces.push_back({i, 0, len, 0});
      continue;
    }
    if (hd.h > 0) pieces.push_back({i, 0, std::min(hd.h, len), 0});
    if (len > hd.h) pieces.push_back({i, hd.h, len - hd.h, hd.level});
  }
  // Total cost, counting the overhead of every item the cuts can add (one
  // per CTA boundary plus the kMaxItem splits): overestimating only leaves
  // the last CTA a little short, underestimating would make it a straggler.
  const double bpe = bytes_per_elem(d);
  double total = kItemOverhead * (grid - 1);
  for (const Piece& p : pieces)
    total += p.n * bpe + kItemOverhead * double((p.n + kMaxItem - 1) / kMaxItem);
  const double quota = total / grid;

  items.clear();
  cta_begin.assign(grid + 1, 0);
  int b = 1;
  double acc = 0;
  for (const Piece& pc : pieces) {
    int64_t off = pc.offset, left = pc.n;
    while (left > 0) {
      int64_t take = std::min(left, kMaxItem);
      if (b < grid) {
        const double room = quota * b - acc;
        if (take * bpe + kItemOverhead > room) {
          int64_t k = static_cast<int64_t>((room - kItemOverhead) / bpe);
          k = k / kCutQuantum * kCutQuantum;
          if (k <= 0) {  // nothing more fits in this CTA: close it
            cta_begin[b++] = static_cast<int32_t>(items.size());
            continue;
          }
          take = std::min(take, k);
        }
      }
      items.push_back({pc.tensor, off, take, pc.level});
      acc += take * bpe + kItemOverhead;
      off += take;
      left -= take;
      while (b < grid && acc >= quota * b) cta_begin[b++] = static_cast<int32_t>(items.size());
    }
  }
  while (b <= grid) cta_begin[b++] = static_cast<int32_t>(items.size());
  cta_begin[grid] = static_cast<int32_t>(items.size());
}

int choose_grid(double total_cost, int grid_max) {
  const double want = std::ceil(total_cost / kMinCtaCost);
  return static_cast<int>(std::max(1.0, std::min(want, static_cast<double>(grid_max))));
}

double total_cost(const fadam_tensor* ts, int64_t n, const Dtypes& d) {
  double c = 0;
  const double bpe = bytes_per_elem(d);
  for (int64_t i = 0; i < n; ++i)
    if (ts[i].numel > 0) c += ts[i].numel * bpe + kItemOverhead;
  return c;
}

Item to_item(const fadam_tensor& t, const PackItem& pi, const Dtypes& d) {
  auto adv = [&](const void* ptr, int esz) -> void* {
    return ptr ? const_cast<char*>(static_cast<const char*>(ptr)) + pi.offset * esz : nullptr;
  };
  Item it;
  it.p = adv(t.p, elem_size(d.p));
  it.m = adv(t.m, mv_size(d));
  it.v = adv(t.v, mv_size(d));
  it.g = adv(t.g, elem_size(d.g));
  it.p_out = adv(t.p_out, elem_size(d.out));
  it.rem = static_cast<int16_t*>(adv(t.rem, 2));
  it.n = static_cast<int32_t>(pi.n);
  it.group = static_cast<uint16_t>(t.group);
  it.flags = static_cast<uint16_t>((pi.level >= 1 ? kItemVec : 0) | (pi.level >= 2 ? kItemBulk : 0));
  it.tensor = static_cast<int32_t>(pi.tensor);
  return it;
}

KernelEntry select_kernel(const Dtypes& d, bool scaled, bool recip) {
  // the remainder form keeps fp32 m and v: its kernels sit with fp32 state
  const int32_t st = d.rem ? FADAM_DT_F32 : d.p;
  const int key = st * 4 + d.g;
  // the reciprocal bias corrections have instances for the 16-bit state
  // forms only
  if (recip && !d.rem && d.mv == FADAM_DT_NONE && st != FADAM_DT_F32) {
    switch (key) {
#define FADAM_RECIP_PICK(S, SD, G, GD)                                                  \
      case SD * 4 + GD:                                                                  \
        return scaled ? recip_scaled_kernel_s##S##_g##G(d.out)                           \
                      : recip_kernel_s##S##_g##G(d.out);
      FADAM_RECIP_PICK(bf16, FADAM_DT_BF16, f32, FADAM_DT_F32)
      FADAM_RECIP_PICK(bf16, FADAM_DT_BF16, bf16, FADAM_DT_BF16)
      FADAM_RECIP_PICK(bf16, FADAM_DT_BF16, f16, FADAM_DT_F16)
      FADAM_RECIP_PICK(f16, FADAM_DT_F16, f32, FADAM_DT_F32)
      FADAM_RECIP_PICK(f16, FADAM_DT_F16, bf16, FADAM_DT_BF16)
      FADAM_RECIP_PICK(f16, FADAM_DT_F16, f16, FADAM_DT_F16)
#undef FADAM_RECIP_PICK
      default: return {nullptr, 0};
    }
  }
  if (d.mv == FADAM_DT_BF16) {
    switch (d.g) {
      case FADAM_DT_F32: return kernel_sf32mbf16_gf32(d.out, false);
      case FADAM_DT_BF16: return kernel_sf32mbf16_gbf16(d.out, false);
      case FADAM_DT_F16: return kernel_sf32mbf16_gf16(d.out, false);
      default: return {nullptr, 0};
    }
  }
  if (d.mv == FADAM_DT_F16) {
    switch (d.g) {
      case FADAM_DT_F32: return kernel_sf32mf16_gf32(d.out, false);
      case FADAM_DT_BF16: return kernel_sf32mf16_gbf16(d.out, false);
      case FADAM_DT_F16: return kernel_sf32mf16_gf16(d.out, false);
      default: return {nullptr, 0};
    }
  }
  if (scaled) {
    switch (key) {
      case FADAM_DT_BF16 * 4 + FADAM_DT_F32: return scaled_kernel_sbf16_gf32(d.out);
      case FADAM_DT_BF16 * 4 + FADAM_DT_BF16: return scaled_kernel_sbf16_gbf16(d.out);
      case FADAM_DT_BF16 * 4 + FADAM_DT_F16: return scaled_kernel_sbf16_gf16(d.out);
      case FADAM_DT_F16 * 4 + FADAM_DT_F32: return scaled_kernel_sf16_gf32(d.out);
      case FADAM_DT_F16 * 4 + FADAM_DT_BF16: return scaled_kernel_sf16_gbf16(d.out);
      case FADAM_DT_F16 * 4 + FADAM_DT_F16: return scaled_kernel_sf16_gf16(d.out);
      default: return {nullptr, 0};
    }
  }
  switch (key) {
    case FADAM_DT_F32 * 4 + FADAM_DT_F32: return kernel_sf32_gf32(d.out, d.rem);
    case FADAM_DT_F32 * 4 + FADAM_DT_BF16: return kernel_sf32_gbf16(d.out, d.rem);
    case FADAM_DT_F32 * 4 + FADAM_DT_F16: return kernel_sf32_gf16(d.out, d.rem);
    case FADAM_DT_BF16 * 4 + FADAM_DT_F32: return kernel_sbf16_gf32(d.out, d.rem);
    case FADAM_DT_BF16 * 4 + FADAM_DT_BF16: return kernel_sbf16_gbf16(d.out, d.rem);
    case FADAM_DT_BF16 * 4 + FADAM_DT_F16: return kernel_sbf16_gf16(d.out, d.rem);
    case FADAM_DT_F16 * 4 + FADAM_DT_F32: return kernel_sf16_gf32(d.out, d.rem);
    case FADAM_DT_F16 * 4 + FADAM_DT_BF16: return kernel_sf16_gbf16(d.out, d.rem);
    case FADAM_DT_F16 * 4 + FADAM_DT_F16: return kernel_sf16_gf16(d.out, d.rem);
    default: return {nullptr, 0};
  }
}

KGroup to_kgroup(const fadam_group& g, bool owns_step) {
  KGroup k{};
  k.beta1 = g.beta1;
  k.beta2 = g.beta2;
  k.eps = g.eps;
  k.wd = g.weight_decay;
  k.lr = g.lr;
  k.grad_scale = g.grad_scale;
  k.step = g.step;
  k.bits = (g.mode == FADAM_MODE_ADAMW ? kGroupAdamW : 0u) |
           (g.bias_correction ? kGroupBiasCorr : 0u) | (owns_step ? kGroupOwnsStep : 0u);
  k.lr_dev = g.lr_dev;
  k.gs_dev = g.grad_scale_dev;
  k.step_dev = g.step_dev;
  return k;
}

// A group owns its step counter when no earlier group uses the same pointer.
void fill_kgroups(const fadam_group* groups, int32_t n_groups, uint32_t flags, KGroup* out) {
  const bool capt = flags & FADAM_CAPTURABLE;
  for (int32_t i = 0; i < n_groups; ++i) {
    bool owns = capt;
    for (int32_t j = 0; j < i && owns; ++j)
      if (groups[j].step_dev == groups[i].step_dev) owns = false;
    out[i] = to_kgroup(groups[i], owns);
  }
}

// Chunks of bulk tiles for the dynamically shared bulk pass, in the order
// the CTAs take them: kChunkTiles tiles each (or more when that keeps the
// list within max_chunks), tapering towards the end of the list so that the
// CTAs finish together: a chunk that starts with R tiles left in the list
// gets about R / (2 grid) of them, down to kTaperMinTiles (guided
// self-scheduling; smaller chunks would leave the g-only passes, which
// read a chunk in tiles of 4-8 update tiles' worth of g, with partial
// tiles).  The tapered list is used when it fits max_chunks.  An item is
// bulk-copied when every stream is 16-byte aligned (kItemBulk); its tiles
// cover its vectors rounded down to an even count.
void build_chunks(const std::vector<Item>& items, int64_t max_chunks, int grid,
                  std::vector<Chunk>& chunks) {
  int64_t total_tiles = 0;
  auto tiles_of = [](const Item& it) -> int64_t {
    if (!(it.flags & kItemBulk)) return 0;
    const int64_t bv = (it.n / kVec) & ~int64_t(1);
    return (bv + kBlock - 1) / kBlock;
  };
  for (const Item& it : items) total_tiles += tiles_of(it);
  int64_t per = kChunkTiles;
  // every item with tiles needs at least one chunk of its own
  int64_t bulk_items = 0;
  for (const Item& it : items) bulk_items += tiles_of(it) > 0;
  const int64_t budget = std::max<int64_t>(1, max_chunks - bulk_items);
  per = std::max<int64_t>(per, (total_tiles + budget - 1) / budget);
  for (int taper = 1; taper >= 0; --taper) {
    chunks.clear();
    int64_t left = total_tiles;  // tiles from the next chunk to the end
    for (size_t k = 0; k < items.size(); ++k) {
      const int64_t nt = tiles_of(items[k]);
      for (int64_t t = 0; t < nt;) {
        int64_t size = per;
        if (taper) size = std::min(per, std::max<int64_t>(kTaperMinTiles, left / (2 * int64_t(grid))));
        size = std::min(size, nt - t);
        chunks.push_back(Chunk{static_cast<int32_t>(k), static_cast<int32_t>(t),
                               static_cast<int32_t>(size), 0});
        t += size;
        left -= size;
      }
    }
    if (int64_t(chunks.size()) <= max_chunks) return;
  }
}

struct HostPlan {
  Dtypes d;
  uint32_t flags = 0;
  const void* kernel = nullptr;
  size_t smem = 0;  // dynamic shared memory of a launch
  int device = 0, sm_count = 0, blocks_per_sm = 0, grid = 1;
  std::vector<Item> items;
  std::vector<int32_t> cta_begin;
  std::vector<Chunk> chunks;
  int64_t n_elements = 0;
  double bytes = 0, check_bytes = 0;
  uint32_t shape = 0;  // kNoTails, kAllBulk
};

// Checks, device query and packing shared by fadam_plan_create and
// fadam_step_once.  Allocates no device memory.
fadam_status prepare(const fadam_tensor* tensors, int64_t n_tensors, const fadam_group* groups,
                     int32_t n_groups, const Dtypes& d, uint32_t flags, bool check_host_step,
                     int64_t max_chunks, HostPlan& hp) {
  fadam_status st = check_dtypes(d, flags);
  if (st) return st;
  if (n_groups < 1 || n_groups > FADAM_MAX_GROUPS)
    return fail(FADAM_EINVAL, "n_groups %d outside 1..%d", n_groups, FADAM_MAX_GROUPS);
  std::vector<char> has_tensor(n_groups, 0);
  st = check_tensors(tensors, n_tensors, n_groups, d, has_tensor);
  if (st) return st;
  st = check_groups(groups, n_groups, flags, has_tensor, check_host_step);
  if (st) return st;

  hp.d = d;
  hp.flags = flags;
  const KernelEntry ke =
      select_kernel(d, (flags & FADAM_SCALED_STATES) != 0, (flags & FADAM_RECIP_BC) != 0);
  hp.kernel = ke.fn;
  hp.smem = ke.smem;
  if (!hp.kernel) return fail(FADAM_EDTYPE, "no kernel for this dtype combination");
  cudaError_t e = cudaGetDevice(&hp.device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&hp.sm_count, cudaDevAttrMultiProcessorCount, hp.device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  e = cudaFuncSetAttribute(hp.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(hp.smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dynamic shared memory)");
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&hp.blocks_per_sm, hp.kernel, kBlock, hp.smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (hp.blocks_per_sm < 1) return fail(FADAM_ECUDA, "kernel cannot be resident on this device");

  const double cost = total_cost(tensors, n_tensors, d);
  hp.grid = choose_grid(cost, hp.blocks_per_sm * hp.sm_count);
  std::vector<PackItem> pitems;
  pack(tensors, n_tensors, d, hp.grid, pitems, hp.cta_begin);
  if (pitems.size() > size_t(INT32_MAX))
    return fail(FADAM_ELIMIT, "more than 2^31 work items");
  hp.items.reserve(pitems.size());
  for (const PackItem& pi : pitems) hp.items.push_back(to_item(tensors[pi.tensor], pi, d));
  build_chunks(hp.items, max_chunks, hp.grid, hp.chunks);
  // a bulk item takes a multiple of 8 elements through the tiles and the
  // rest element-wise in the tail pass
  hp.shape = kNoTails | kAllBulk;
  for (const Item& it : hp.items) {
    if (!(it.flags & kItemBulk)) hp.shape &= ~kAllBulk;
    else if (it.n % 8 != 0) hp.shape &= ~kNoTails;
  }
  const double bpe = bytes_per_elem(d);
  for (int64_t i = 0; i < n_tensors; ++i) {
    const int64_t ne = std::max<int64_t>(tensors[i].numel, 0);
    hp.n_elements += ne;
    double b = ne * bpe;
    // a param-out that aliases the master (same dtype) is the same stream
    if (!d.rem && tensors[i].p_out && tensors[i].p_out == tensors[i].p) b -= ne * double(elem_size(d.out));
    hp.bytes += b;
  }
  if (flags & FADAM_CHECK_FINITE) hp.check_bytes = hp.n_elements * double(elem_size(d.g));
  return FADAM_OK;
}

fadam_status launch(const void* kernel, size_t smem, const KParams& kp, int grid, bool cooperative,
                    cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (cooperative) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[1] = {const_cast<KParams*>(&kp)};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return FADAM_OK;
}

}  // namespace

struct fadam_plan {
  HostPlan hp;
  std::vector<fadam_tensor> tensors;
  std::vector<fadam_group> groups;
  std::vector<char> has_tensor;
  int32_t n_groups = 0;
  Item* d_items = nullptr;
  Chunk* d_chunks = nullptr;
  int32_t* d_cta = nullptr;
  KScratch* d_scratch = nullptr;
  BcMemo* d_memo = nullptr;      // bias corrections carried from one launch to the next
  double* d_partials = nullptr;  // gradient-norm launches: per-chunk and per-item partials
  // the data-parallel exchange (fadam_plan_set_exchange): byte offsets
  int32_t n_sources = 0, average = 0, n_dests = 0;
  int64_t src_delta[FADAM_MAX_SOURCES] = {};
  int64_t dst_delta[FADAM_MAX_DESTS] = {};
  // scaled state: the caller's scales and the plan's absmax workspace
  float* scales = nullptr;
  unsigned* d_absmax = nullptr;
  // host-gradient steps: per tensor its device g, and the host gradient's
  // device-accessible address (written by each call)
  const char** d_dev_g = nullptr;
  const char** d_host_g = nullptr;
  std::vector<const char*> host_g;
  // FADAM_TEST_BARRIER_TIMEOUT acts on the plan's first step launch only
  bool test_timeout_armed = false;
};

namespace {

void free_plan_memory(fadam_plan* p) {
  if (p->d_absmax) cudaFree(p->d_absmax);
  p->d_absmax = nullptr;
  if (p->d_dev_g) cudaFree(p->d_dev_g);
  if (p->d_host_g) cudaFree(p->d_host_g);
  p->d_dev_g = p->d_host_g = nullptr;
  if (p->d_items) cudaFree(p->d_items);
  if (p->d_chunks) cudaFree(p->d_chunks);
  if (p->d_cta) cudaFree(p->d_cta);
  if (p->d_scratch) cudaFree(p->d_scratch);
  if (p->d_memo) cudaFree(p->d_memo);
  if (p->d_partials) cudaFree(p->d_partials);
  p->d_items = nullptr;
  p->d_chunks = nullptr;
  p->d_cta = nullptr;
  p->d_scratch = nullptr;
  p->d_partials = nullptr;
}

void fill_params(KParams& kp, const Item* items, const int32_t* cta, const Chunk* chunks,
                 int32_t n_chunks, int32_t* noop, KScratch* scratch, const fadam_group* groups,
                 int32_t n_groups, uint32_t flags) {
  memset(&kp, 0, sizeof kp);
  kp.items = items;
  kp.cta_begin = cta;
  kp.chunks = chunks;
  kp.n_chunks = n_chunks;
  kp.noop = noop;
  kp.scratch = scratch;
  kp.n_groups = n_groups;
  kp.flags = flags;
  fill_kgroups(groups, n_groups, flags, kp.groups);
}

void fill_scaled(KParams& kp, const fadam_plan* plan) {
  if (!(plan->hp.flags & FADAM_SCALED_STATES)) return;
  kp.scales = plan->scales;
  kp.absmax = plan->d_absmax;
  kp.n_tensors = static_cast<int32_t>(plan->tensors.size());
  // half the largest finite value of the state dtype
  kp.max_scaled = plan->hp.d.p == FADAM_DT_F16 ? 0x1.ffcp+14f   // 65504 / 2
                                                : 0x1.fep+126f;  // 0x7F7F as bf16, / 2
}

void fill_exchange(KParams& kp, const fadam_plan* plan) {
  kp.n_sources = plan->n_sources;
  kp.average = plan->average;
  kp.n_dests = plan->n_dests;
  const int r_n = plan->n_sources;
  kp.avg_mul = ((plan->average & FADAM_EXCHANGE_AVERAGE) && r_n > 0 && (r_n & (r_n - 1)) == 0)
                   ? 1.0f / static_cast<float>(r_n)
                   : 0.0f;
  for (int r = 0; r < plan->n_sources; ++r) kp.src_delta[r] = plan->src_delta[r];
  for (int d = 0; d < plan->n_dests; ++d) kp.dst_delta[d] = plan->dst_delta[d];
}

// The plan's flags for a step launch: the barrier-timeout diagnostic goes
// to the first such launch only, so that the launches after it show that a
// plan recovers from a wait that gave up.
uint32_t step_flags(fadam_plan* plan) {
  uint32_t f = plan->hp.flags & ~kTestBarrierTimeout;
  if (plan->test_timeout_armed) {
    f |= kTestBarrierTimeout;
    plan->test_timeout_armed = false;
  }
  return f;
}

bool needs_launch(const HostPlan& hp) {
  const bool owns_steps = (hp.flags & FADAM_CAPTURABLE) && !(hp.flags & FADAM_STEP_PREADVANCED);
  return !hp.items.empty() || owns_steps;
}

}  // namespace

extern "C" {

fadam_status fadam_plan_create(const fadam_tensor* tensors, int64_t n_tensors,
                               const fadam_group* groups, int32_t n_groups, int32_t p_dtype,
                               int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                               fadam_plan** plan_out) {
  t_last_error.clear();
  if (!plan_out) return fail(FADAM_EINVAL, "plan_out is NULL");
  *plan_out = nullptr;
  const Dtypes d = make_dtypes(p_dtype, g_dtype, out_dtype, flags);
  fadam_plan* plan = new (std::nothrow) fadam_plan();
  if (!plan) return fail(FADAM_EINVAL, "out of host memory");
  // the host step of a regular plan is per-step data: checked at launch
  fadam_status st = prepare(tensors, n_tensors, groups, n_groups, d, flags, false, kPlanMaxChunks,
                            plan->hp);
  if (st) {
    delete plan;
    return st;
  }
  plan->tensors.assign(tensors, tensors + n_tensors);
  plan->groups.assign(groups, groups + n_groups);
  plan->n_groups = n_groups;
  plan->test_timeout_armed = (flags & FADAM_TEST_BARRIER_TIMEOUT) != 0;
  const HostPlan& hp = plan->hp;
  cudaError_t e = cudaSuccess;
  if (!hp.items.empty()) {
    e = cudaMalloc(&plan->d_items, hp.items.size() * sizeof(Item));
    if (e == cudaSuccess)
      e = cudaMemcpy(plan->d_items, hp.items.data(), hp.items.size() * sizeof(Item),
                     cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && !hp.chunks.empty()) {
    e = cudaMalloc(&plan->d_chunks, hp.chunks.size() * sizeof(Chunk));
    if (e == cudaSuccess)
      e = cudaMemcpy(plan->d_chunks, hp.chunks.data(), hp.chunks.size() * sizeof(Chunk),
                     cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_cta, hp.cta_begin.size() * sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaMemcpy(plan->d_cta, hp.cta_begin.data(), hp.cta_begin.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_scratch, sizeof(KScratch));
  if (e == cudaSuccess) e = cudaMemset(plan->d_scratch, 0, sizeof(KScratch));
  // no memo entry is valid until a launch writes it (tag 0)
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_memo, kMemoEntries * sizeof(BcMemo));
  if (e == cudaSuccess) e = cudaMemset(plan->d_memo, 0, kMemoEntries * sizeof(BcMemo));
  // gradient-norm launches: one partial per tile chunk and per item
  if (e == cudaSuccess)
    e = cudaMalloc(&plan->d_partials, (hp.chunks.size() + hp.items.size() + 1) * sizeof(double));
  // host-gradient steps: the tensors' device g pointers, and room for the
  // host ones
  if (e == cudaSuccess && n_tensors > 0) {
    std::vector<const char*> dev_g(n_tensors);
    for (int64_t i = 0; i < n_tensors; ++i) dev_g[i] = static_cast<const char*>(tensors[i].g);
    e = cudaMalloc(&plan->d_dev_g, size_t(n_tensors) * sizeof(char*));
    if (e == cudaSuccess)
      e = cudaMemcpy(plan->d_dev_g, dev_g.data(), size_t(n_tensors) * sizeof(char*),
                     cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc(&plan->d_host_g, size_t(n_tensors) * sizeof(char*));
    plan->host_g.assign(size_t(n_tensors), nullptr);
  }
  // scaled state: three absmax slots per tensor, zero between steps
  if (e == cudaSuccess && (flags & FADAM_SCALED_STATES) && n_tensors > 0) {
    e = cudaMalloc(&plan->d_absmax, size_t(n_tensors) * 3 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(plan->d_absmax, 0, size_t(n_tensors) * 3 * sizeof(unsigned));
  }
  if (e != cudaSuccess) {
    st = cuda_fail(e, "plan upload");
    free_plan_memory(plan);
    delete plan;
    return st;
  }
  *plan_out = plan;
  return FADAM_OK;
}

fadam_status fadam_plan_set_groups(fadam_plan* plan, const fadam_group* groups, int32_t n_groups) {
  t_last_error.clear();
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (n_groups != plan->n_groups)
    return fail(FADAM_EINVAL, "n_groups %d differs from the plan's %d", n_groups, plan->n_groups);
  std::vector<char> has_tensor(n_groups, 0);
  for (const fadam_tensor& t : plan->tensors)
    if (t.numel > 0) has_tensor[t.group] = 1;
  const fadam_status st = check_groups(groups, n_groups, plan->hp.flags, has_tensor, false);
  if (st) return st;
  plan->groups.assign(groups, groups + n_groups);
  return FADAM_OK;
}

namespace {
fadam_status step_launch(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream,
                         uint32_t extra_flags);
}  // namespace

fadam_status fadam_step(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream) {
  return step_launch(plan, noop_dev, stream, 0u);
}

namespace {
fadam_status step_launch(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream,
                         uint32_t extra_flags) {
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  const HostPlan& hp = plan->hp;
  if ((hp.flags & FADAM_CHECK_FINITE) && !noop_dev)
    return fail(FADAM_EINVAL, "FADAM_CHECK_FINITE needs a noop_dev flag to write");
  if (noop_dev && reinterpret_cast<uintptr_t>(noop_dev) % 4)
    return fail(FADAM_EALIGN, "noop_dev is not 4-byte aligned");
  if (!needs_launch(hp)) return FADAM_OK;
  if (!(hp.flags & FADAM_CAPTURABLE))
    for (int32_t i = 0; i < plan->n_groups; ++i)
      if (plan->groups[i].bias_correction == 1 && plan->groups[i].step < 1)
        return fail(FADAM_EINVAL, "group %d: step %d < 1 with bias correction (1-beta^step = 0)",
                    i, plan->groups[i].step);
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  const bool scaled = (hp.flags & FADAM_SCALED_STATES) != 0;
  if (scaled && !plan->scales)
    return fail(FADAM_EINVAL, "a scaled-state plan needs fadam_plan_set_state_scales first");
  KParams kp;
  fill_params(kp, plan->d_items, plan->d_cta, plan->d_chunks, static_cast<int32_t>(hp.chunks.size()),
              noop_dev, plan->d_scratch, plan->groups.data(), plan->n_groups,
              step_flags(plan) | hp.shape | extra_flags);
  fill_exchange(kp, plan);
  fill_scaled(kp, plan);
  kp.memo = plan->d_memo;
  kp.n_sources = 0;  // the plain step reads g as it stands
  kp.host_g = plan->d_host_g;
  kp.dev_g = plan->d_dev_g;
  return launch(hp.kernel, hp.smem, kp, hp.grid, (hp.flags & FADAM_CHECK_FINITE) != 0 || scaled,
                reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

fadam_status fadam_plan_set_state_scales(fadam_plan* plan, float* scales_dev) {
  t_last_error.clear();
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (!(plan->hp.flags & FADAM_SCALED_STATES))
    return fail(FADAM_EINVAL, "the plan was not created with FADAM_SCALED_STATES");
  if (!scales_dev) return fail(FADAM_EINVAL, "scales_dev is NULL");
  if (reinterpret_cast<uintptr_t>(scales_dev) % 4)
    return fail(FADAM_EALIGN, "scales_dev is not 4-byte aligned");
  plan->scales = scales_dev;
  return FADAM_OK;
}

fadam_status fadam_plan_set_exchange(fadam_plan* plan, const void* g_shard,
                                     const void* const* sources, int32_t n_sources,
                                     int32_t reduce_flags, const void* out_shard,
                                     void* const* dests, int32_t n_dests) {
  t_last_error.clear();
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (n_sources < 0 || n_sources > FADAM_MAX_SOURCES)
    return fail(FADAM_EINVAL, "n_sources %d outside 0..%d", n_sources, FADAM_MAX_SOURCES);
  if (n_dests < 0 || n_dests > FADAM_MAX_DESTS)
    return fail(FADAM_EINVAL, "n_dests %d outside 0..%d", n_dests, FADAM_MAX_DESTS);
  if (reduce_flags & ~(FADAM_EXCHANGE_AVERAGE | FADAM_EXCHANGE_ACCUMULATE))
    return fail(FADAM_EINVAL, "reduce_flags 0x%x: only FADAM_EXCHANGE_AVERAGE and "
                              "FADAM_EXCHANGE_ACCUMULATE are defined", reduce_flags);
  int64_t src[FADAM_MAX_SOURCES] = {}, dst[FADAM_MAX_DESTS] = {};
  if (n_sources > 0) {
    if (!g_shard || !sources) return fail(FADAM_EINVAL, "g_shard and sources are needed");
    for (int32_t r = 0; r < n_sources; ++r) {
      if (!sources[r]) return fail(FADAM_EINVAL, "sources[%d] is NULL", r);
      src[r] = static_cast<int64_t>(reinterpret_cast<uintptr_t>(sources[r]) -
                                    reinterpret_cast<uintptr_t>(g_shard));
      if (src[r] % 16) return fail(FADAM_EALIGN, "sources[%d] - g_shard is not a multiple of 16 bytes", r);
    }
  }
  if (n_dests > 0) {
    if (plan->hp.d.out == FADAM_DT_NONE && !plan->hp.d.rem)
      return fail(FADAM_EINVAL, "exchange destinations need a param-out dtype");
    if (!out_shard || !dests) return fail(FADAM_EINVAL, "out_shard and dests are needed");
    for (int32_t d = 0; d < n_dests; ++d) {
      if (!dests[d]) return fail(FADAM_EINVAL, "dests[%d] is NULL", d);
      dst[d] = static_cast<int64_t>(reinterpret_cast<uintptr_t>(dests[d]) -
                                    reinterpret_cast<uintptr_t>(out_shard));
      if (dst[d] % 16) return fail(FADAM_EALIGN, "dests[%d] - out_shard is not a multiple of 16 bytes", d);
    }
  }
  plan->n_sources = n_sources;
  plan->average = reduce_flags;
  plan->n_dests = n_dests;
  for (int r = 0; r < FADAM_MAX_SOURCES; ++r) plan->src_delta[r] = src[r];
  for (int d = 0; d < FADAM_MAX_DESTS; ++d) plan->dst_delta[d] = dst[d];
  return FADAM_OK;
}

fadam_status fadam_grad_reduce(fadam_plan* plan, fadam_stream stream) {
  t_last_error.clear();
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (plan->n_sources < 1) return fail(FADAM_EINVAL, "no exchange sources set");
  const HostPlan& hp = plan->hp;
  if (hp.items.empty()) return FADAM_OK;
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  KParams kp;
  fill_params(kp, plan->d_items, plan->d_cta, plan->d_chunks, static_cast<int32_t>(hp.chunks.size()),
              nullptr, plan->d_scratch, plan->groups.data(), plan->n_groups,
              (hp.flags & FADAM_CAPTURABLE) | hp.shape | kReduceOnly);
  fill_exchange(kp, plan);
  return launch(hp.kernel, hp.smem, kp, hp.grid, false, reinterpret_cast<cudaStream_t>(stream));
}

fadam_status fadam_step_reduce(fadam_plan* plan, int32_t* noop_dev, fadam_stream stream) {
  t_last_error.clear();
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (plan->n_sources < 1) return fail(FADAM_EINVAL, "no exchange sources set");
  const HostPlan& hp = plan->hp;
  if ((hp.flags & FADAM_CHECK_FINITE) && !noop_dev)
    return fail(FADAM_EINVAL, "FADAM_CHECK_FINITE needs a noop_dev flag to write");
  if (noop_dev && reinterpret_cast<uintptr_t>(noop_dev) % 4)
    return fail(FADAM_EALIGN, "noop_dev is not 4-byte aligned");
  if (!needs_launch(hp)) return FADAM_OK;
  if (!(hp.flags & FADAM_CAPTURABLE))
    for (int32_t i = 0; i < plan->n_groups; ++i)
      if (plan->groups[i].bias_correction == 1 && plan->groups[i].step < 1)
        return fail(FADAM_EINVAL, "group %d: step %d < 1 with bias correction (1-beta^step = 0)",
                    i, plan->groups[i].step);
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  if ((hp.flags & FADAM_SCALED_STATES) && !plan->scales)
    return fail(FADAM_EINVAL, "a scaled-state plan needs fadam_plan_set_state_scales first");
  KParams kp;
  fill_params(kp, plan->d_items, plan->d_cta, plan->d_chunks, static_cast<int32_t>(hp.chunks.size()),
              noop_dev, plan->d_scratch, plan->groups.data(), plan->n_groups,
              step_flags(plan) | hp.shape | kReduceFirst);
  fill_exchange(kp, plan);
  fill_scaled(kp, plan);
  kp.memo = plan->d_memo;
  return launch(hp.kernel, hp.smem, kp, hp.grid, true, reinterpret_cast<cudaStream_t>(stream));
}

fadam_status fadam_step_host_grads(fadam_plan* plan, const void* const* g_host, int32_t* noop_dev,
                                   int32_t* steps_host, fadam_stream stream) {
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  const HostPlan& hp = plan->hp;
  const int gsz = elem_size(hp.d.g);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool any = false;
  for (const fadam_tensor& t : plan->tensors) any |= t.numel > 0;
  if (any && !g_host) return fail(FADAM_EINVAL, "g_host is NULL");
  for (size_t i = 0; i < plan->tensors.size(); ++i)
    if (plan->tensors[i].numel > 0 && !g_host[i])
      return fail(FADAM_EINVAL, "g_host[%zu] is NULL", i);
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  // zero copy when every host gradient is page-locked and mapped for this
  // device: the update reads it over the host link itself, so the transfer
  // and the update of the other streams overlap
  bool mapped = any && plan->d_host_g != nullptr;
  for (size_t i = 0; mapped && i < plan->tensors.size(); ++i) {
    plan->host_g[i] = nullptr;
    if (plan->tensors[i].numel <= 0) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, g_host[i]) != cudaSuccess || a.type != cudaMemoryTypeHost ||
        a.devicePointer == nullptr || reinterpret_cast<uintptr_t>(a.devicePointer) % 16 !=
                                          reinterpret_cast<uintptr_t>(plan->tensors[i].g) % 16) {
      cudaGetLastError();  // clear the query's error for unregistered memory
      mapped = false;
      break;
    }
    plan->host_g[i] = static_cast<const char*>(a.devicePointer);
  }
  fadam_status st = FADAM_OK;
  if (mapped) {
    const cudaError_t e = cudaMemcpyAsync(plan->d_host_g, plan->host_g.data(),
                                          plan->host_g.size() * sizeof(char*),
                                          cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "host gradient table upload");
    st = step_launch(plan, noop_dev, stream, kHostGrads);
  } else {
    for (size_t i = 0; i < plan->tensors.size(); ++i) {
      const fadam_tensor& t = plan->tensors[i];
      if (t.numel <= 0) continue;
      const cudaError_t e = cudaMemcpyAsync(const_cast<void*>(t.g), g_host[i],
                                            size_t(t.numel) * gsz, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "gradient upload");
    }
    st = fadam_step(plan, noop_dev, stream);
  }
  if (st) return st;
  if (steps_host) {
    for (int32_t g = 0; g < plan->n_groups; ++g) {
      const fadam_group& gr = plan->groups[g];
      if (hp.flags & FADAM_CAPTURABLE) {
        const cudaError_t e =
            cudaMemcpyAsync(&steps_host[g], gr.step_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "step counter read");
      } else {
        steps_host[g] = gr.step;
      }
    }
  }
  const cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return FADAM_OK;
}

fadam_status fadam_plan_status(fadam_plan* plan, int32_t* device_status) {
  if (!plan || !device_status) return fail(FADAM_EINVAL, "plan or device_status is NULL");
  DeviceGuard guard(plan->hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  KScratch sc;
  cudaError_t e = cudaMemcpy(&sc, plan->d_scratch, sizeof sc, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *device_status = sc.status;
  if (sc.status != FADAM_OK || sc.bar_count != 0 || sc.done != 0) {
    e = cudaMemset(plan->d_scratch, 0, sizeof(KScratch));
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
  }
  return FADAM_OK;
}

fadam_status fadam_plan_get_info(const fadam_plan* plan, fadam_plan_info* info) {
  if (!plan || !info) return fail(FADAM_EINVAL, "plan or info is NULL");
  const HostPlan& hp = plan->hp;
  memset(info, 0, sizeof *info);
  info->n_tensors = static_cast<int64_t>(plan->tensors.size());
  info->n_elements = hp.n_elements;
  info->n_items = static_cast<int64_t>(hp.items.size());
  info->n_chunks = static_cast<int64_t>(hp.chunks.size());
  info->grid = hp.grid;
  info->block = kBlock;
  info->blocks_per_sm = hp.blocks_per_sm;
  info->sm_count = hp.sm_count;
  info->n_groups = plan->n_groups;
  info->device = hp.device;
  info->bytes_per_step = hp.bytes;
  info->check_bytes_per_step = hp.check_bytes;
  return FADAM_OK;
}

fadam_status fadam_plan_destroy(fadam_plan* plan) {
  if (!plan) return FADAM_OK;
  {
    DeviceGuard guard(plan->hp.device);
    free_plan_memory(plan);
  }
  delete plan;
  return FADAM_OK;
}

fadam_status fadam_step_once(const fadam_tensor* tensors, int64_t n_tensors, int32_t mode,
                             int32_t bias_correction, float beta1, float beta2, float eps,
                             float weight_decay, float lr, const float* lr_dev, int32_t step,
                             int32_t* step_dev, float grad_scale, const float* grad_scale_dev,
                             int32_t* noop_dev, int32_t g_dtype, int32_t out_dtype,
                             fadam_stream stream) {
  t_last_error.clear();
  const int n_dev = (lr_dev != nullptr) + (step_dev != nullptr) + (grad_scale_dev != nullptr);
  if (n_dev != 0 && n_dev != 3)
    return fail(FADAM_EINVAL, "give all of lr_dev, step_dev, grad_scale_dev or none");
  const uint32_t flags = n_dev == 3 ? FADAM_CAPTURABLE : 0u;
  fadam_group grp{};
  grp.mode = mode;
  grp.bias_correction = bias_correction;
  grp.beta1 = beta1;
  grp.beta2 = beta2;
  grp.eps = eps;
  grp.weight_decay = weight_decay;
  grp.lr = lr;
  grp.grad_scale = grad_scale;
  grp.step = step;
  grp.lr_dev = lr_dev;
  grp.grad_scale_dev = grad_scale_dev;
  grp.step_dev = step_dev;
  for (int64_t i = 0; i < n_tensors && tensors; ++i)
    if (tensors[i].group != 0) return fail(FADAM_EINVAL, "one-shot tensors must all be group 0");
  if (noop_dev && reinterpret_cast<uintptr_t>(noop_dev) % 4)
    return fail(FADAM_EALIGN, "noop_dev is not 4-byte aligned");
  HostPlan hp;
  const Dtypes d{FADAM_DT_F32, g_dtype, out_dtype, false};
  fadam_status st = prepare(tensors, n_tensors, &grp, 1, d, flags, true, kPlanMaxChunks, hp);
  if (st) return st;
  if (!needs_launch(hp)) return FADAM_OK;
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Item* d_items = nullptr;
  Chunk* d_chunks = nullptr;
  int32_t* d_cta = nullptr;
  KScratch* d_scratch = nullptr;
  cudaError_t e = cudaSuccess;
  if (!hp.items.empty()) {
    e = cudaMallocAsync(&d_items, hp.items.size() * sizeof(Item), s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(d_items, hp.items.data(), hp.items.size() * sizeof(Item),
                          cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess && !hp.chunks.empty()) {
    e = cudaMallocAsync(&d_chunks, hp.chunks.size() * sizeof(Chunk), s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(d_chunks, hp.chunks.data(), hp.chunks.size() * sizeof(Chunk),
                          cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess) e = cudaMallocAsync(&d_cta, hp.cta_begin.size() * sizeof(int32_t), s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_cta, hp.cta_begin.data(), hp.cta_begin.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMallocAsync(&d_scratch, sizeof(KScratch), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_scratch, 0, sizeof(KScratch), s);
  if (e == cudaSuccess) {
    KParams kp;
    fill_params(kp, d_items, d_cta, d_chunks, static_cast<int32_t>(hp.chunks.size()), noop_dev,
                d_scratch, &grp, 1, flags | hp.shape);
    st = launch(hp.kernel, hp.smem, kp, hp.grid, false, s);
  } else {
    st = cuda_fail(e, "one-shot upload");
  }
  if (d_items) cudaFreeAsync(d_items, s);
  if (d_chunks) cudaFreeAsync(d_chunks, s);
  if (d_cta) cudaFreeAsync(d_cta, s);
  if (d_scratch) cudaFreeAsync(d_scratch, s);
  return st;
}

}  // extern "C"

namespace {

struct ClipArgs {
  const double* sumsq;
  float* norm_out;
  int32_t* noop;
  float max_norm;
  int32_t n_scales;
  float* scales[FADAM_MAX_GROUPS];
  // regular plans: each group's host grad_scale in, the clipped one out
  int32_t n_host;
  float* host_out;
  float host_in[FADAM_MAX_GROUPS];
};

// One thread: the norm from the squared norm, found_inf into the noop flag,
// and the clip coefficient multiplied into each distinct device grad_scale
// (capturable plans) or into each group's host grad_scale, written out for
// the caller to keep (regular plans).
__global__ void fadam_clip_kernel(const __grid_constant__ ClipArgs a) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const float norm = __double2float_rn(sqrt(__ldcg(a.sumsq)));
  if (a.norm_out) *a.norm_out = norm;
  if (a.noop) *a.noop = isfinite(norm) ? 0 : 1;
  float coef = 1.0f;
  if (a.max_norm > 0.0f) {
    coef = __fdiv_rn(a.max_norm, __fadd_rn(norm, 1e-6f));
    if (coef > 1.0f) coef = 1.0f;  // a NaN coefficient stays NaN, as torch.clamp keeps it
    for (int i = 0; i < a.n_scales; ++i) *a.scales[i] = __fmul_rn(*a.scales[i], coef);
  }
  for (int i = 0; i < a.n_host; ++i)
    a.host_out[i] = a.max_norm > 0.0f ? __fmul_rn(a.host_in[i], coef) : a.host_in[i];
}

}  // namespace

extern "C" {

fadam_status fadam_grad_sumsq(fadam_plan* plan, double* sumsq_dev, fadam_stream stream) {
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (!sumsq_dev || reinterpret_cast<uintptr_t>(sumsq_dev) % 8)
    return fail(FADAM_EINVAL, "sumsq_dev must be a non-NULL, 8-byte aligned device pointer");
  const HostPlan& hp = plan->hp;
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  KParams kp;
  fill_params(kp, plan->d_items, plan->d_cta, plan->d_chunks, static_cast<int32_t>(hp.chunks.size()),
              nullptr, plan->d_scratch, plan->groups.data(), plan->n_groups,
              (hp.flags & FADAM_CAPTURABLE) | hp.shape | kNormOnly);
  kp.partials = plan->d_partials;
  kp.sumsq_out = sumsq_dev;
  return launch(hp.kernel, hp.smem, kp, hp.grid, false, reinterpret_cast<cudaStream_t>(stream));
}

fadam_status fadam_clip_apply(fadam_plan* plan, const double* sumsq_dev, float max_norm,
                              float* norm_dev, int32_t* noop_dev, float* grad_scales_out_dev,
                              fadam_stream stream) {
  if (!plan) return fail(FADAM_EINVAL, "plan is NULL");
  if (!sumsq_dev || reinterpret_cast<uintptr_t>(sumsq_dev) % 8)
    return fail(FADAM_EINVAL, "sumsq_dev must be a non-NULL, 8-byte aligned device pointer");
  if ((norm_dev && reinterpret_cast<uintptr_t>(norm_dev) % 4) ||
      (noop_dev && reinterpret_cast<uintptr_t>(noop_dev) % 4))
    return fail(FADAM_EALIGN, "norm_dev / noop_dev not 4-byte aligned");
  if (grad_scales_out_dev && reinterpret_cast<uintptr_t>(grad_scales_out_dev) % 4)
    return fail(FADAM_EALIGN, "grad_scales_out_dev not 4-byte aligned");
  if (!std::isfinite(max_norm)) return fail(FADAM_EINVAL, "max_norm is not finite");
  ClipArgs a{};
  a.sumsq = sumsq_dev;
  a.norm_out = norm_dev;
  a.noop = noop_dev;
  a.max_norm = max_norm;
  if (plan->hp.flags & FADAM_CAPTURABLE) {
    for (int32_t g = 0; g < plan->n_groups; ++g) {
      float* gs = const_cast<float*>(plan->groups[g].grad_scale_dev);
      if (!gs) continue;
      bool seen = false;
      for (int32_t j = 0; j < a.n_scales; ++j) seen |= a.scales[j] == gs;
      if (!seen) a.scales[a.n_scales++] = gs;
    }
  } else if (grad_scales_out_dev) {
    a.n_host = plan->n_groups;
    a.host_out = grad_scales_out_dev;
    for (int32_t g = 0; g < plan->n_groups; ++g) a.host_in[g] = plan->groups[g].grad_scale;
  }
  DeviceGuard guard(plan->hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  void* args[1] = {&a};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&fadam_clip_kernel), args);
  if (e != cudaSuccess) return cuda_fail(e, "clip kernel launch");
  return FADAM_OK;
}

fadam_status fadam_pack_dry(const fadam_tensor* tensors, int64_t n_tensors, int32_t n_groups,
                            int32_t p_dtype, int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                            int32_t grid, fadam_pack_item* items_out, int64_t max_items,
                            int32_t* cta_begin_out, int64_t* n_items_out) {
  t_last_error.clear();
  const Dtypes d = make_dtypes(p_dtype, g_dtype, out_dtype, flags);
  fadam_status st = check_dtypes(d, flags);
  if (st) return st;
  if (n_groups < 1 || n_groups > FADAM_MAX_GROUPS)
    return fail(FADAM_EINVAL, "n_groups %d outside 1..%d", n_groups, FADAM_MAX_GROUPS);
  std::vector<char> has_tensor(n_groups, 0);
  st = check_tensors(tensors, n_tensors, n_groups, d, has_tensor);
  if (st) return st;
  if (grid < 1) return fail(FADAM_EINVAL, "grid %d < 1", grid);
  if (!n_items_out) return fail(FADAM_EINVAL, "n_items_out is NULL");
  std::vector<PackItem> items;
  std::vector<int32_t> cta;
  pack(tensors, n_tensors, d, grid, items, cta);
  *n_items_out = static_cast<int64_t>(items.size());
  if (cta_begin_out) memcpy(cta_begin_out, cta.data(), cta.size() * sizeof(int32_t));
  if (items_out) {
    if (static_cast<int64_t>(items.size()) > max_items)
      return fail(FADAM_ELIMIT, "%zu items do not fit in max_items %lld", items.size(),
                  (long long)max_items);
    for (size_t i = 0; i < items.size(); ++i) {
      items_out[i].tensor = items[i].tensor;
      items_out[i].offset = items[i].offset;
      items_out[i].n = static_cast<int32_t>(items[i].n);
      items_out[i].vec = items[i].level;
    }
  }
  return FADAM_OK;
}

fadam_status fadam_chunk_dry(const fadam_tensor* tensors, int64_t n_tensors, int32_t n_groups,
                             int32_t p_dtype, int32_t g_dtype, int32_t out_dtype, uint32_t flags,
                             int32_t grid, int64_t max_chunks, int32_t* chunks_out,
                             int64_t max_out, int64_t* n_chunks_out) {
  t_last_error.clear();
  const Dtypes d = make_dtypes(p_dtype, g_dtype, out_dtype, flags);
  fadam_status st = check_dtypes(d, flags);
  if (st) return st;
  if (n_groups < 1 || n_groups > FADAM_MAX_GROUPS)
    return fail(FADAM_EINVAL, "n_groups %d outside 1..%d", n_groups, FADAM_MAX_GROUPS);
  std::vector<char> has_tensor(n_groups, 0);
  st = check_tensors(tensors, n_tensors, n_groups, d, has_tensor);
  if (st) return st;
  if (grid < 1) return fail(FADAM_EINVAL, "grid %d < 1", grid);
  if (max_chunks < 1) return fail(FADAM_EINVAL, "max_chunks %lld < 1", (long long)max_chunks);
  if (!n_chunks_out) return fail(FADAM_EINVAL, "n_chunks_out is NULL");
  std::vector<PackItem> pitems;
  std::vector<int32_t> cta;
  pack(tensors, n_tensors, d, grid, pitems, cta);
  std::vector<Item> items;
  items.reserve(pitems.size());
  for (const PackItem& pi : pitems) items.push_back(to_item(tensors[pi.tensor], pi, d));
  std::vector<Chunk> chunks;
  build_chunks(items, max_chunks, grid, chunks);
  *n_chunks_out = static_cast<int64_t>(chunks.size());
  if (chunks_out) {
    if (static_cast<int64_t>(chunks.size()) > max_out)
      return fail(FADAM_ELIMIT, "%zu chunks do not fit in max_out %lld", chunks.size(),
                  (long long)max_out);
    for (size_t i = 0; i < chunks.size(); ++i) {
      chunks_out[3 * i] = chunks[i].item;
      chunks_out[3 * i + 1] = chunks[i].tile0;
      chunks_out[3 * i + 2] = chunks[i].ntiles;
    }
  }
  return FADAM_OK;
}

const char* fadam_status_string(fadam_status status) {
  switch (status) {
    case FADAM_OK: return "ok";
    case FADAM_EINVAL: return "invalid argument";
    case FADAM_EDTYPE: return "unsupported dtype combination";
    case FADAM_EALIGN: return "misaligned pointer";
    case FADAM_ECUDA: return "CUDA runtime error";
    case FADAM_ETIMEOUT: return "device-side wait timed out";
    case FADAM_ELIMIT: return "size beyond a documented maximum";
    default: return "unknown status";
  }
}

const char* fadam_last_error(void) { return t_last_error.c_str(); }

int32_t fadam_version(void) { return 10000; }

}  // extern "C"

// ---- one-call step without device allocation ----------------------------------
//
// The plan path keeps its work list and status block in memory it allocates
// with cudaMalloc.  fadam_step_noalloc keeps them instead in one file-scope
// device array, g_noalloc_arena, that every GPU loading this library holds
// until the process exits.  Host code never uses the array's name as an
// address: its device address is looked up once per device with
// cudaGetSymbolAddress and handed to the kernel.

#include <mutex>

namespace {

constexpr int64_t kNoAllocMaxItems = 4096;
constexpr int64_t kNoAllocMaxChunks = 4096;
constexpr int32_t kNoAllocMaxCtas = 2048;
constexpr size_t kArenaScratchOff = 0;
constexpr size_t kArenaCtaOff = 256;
constexpr size_t kArenaItemsOff =
    kArenaCtaOff + ((size_t(kNoAllocMaxCtas) + 1) * sizeof(int32_t) + 255) / 256 * 256;
constexpr size_t kArenaChunksOff = kArenaItemsOff + size_t(kNoAllocMaxItems) * sizeof(Item);
constexpr size_t kArenaMemoOff = kArenaChunksOff + size_t(kNoAllocMaxChunks) * sizeof(Chunk);
constexpr size_t kArenaBytes = kArenaMemoOff + size_t(kMemoEntries) * sizeof(BcMemo);
static_assert(sizeof(KScratch) <= kArenaCtaOff, "status block fits its slot");

constexpr int kMaxDevices = 64;
std::mutex g_arena_mutex;
void* g_arena_ptr[kMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_arena[kArenaBytes];

namespace {

// Device address of g_noalloc_arena on `dev` (which must be current),
// looked up on the first call for that device and kept for the life of the
// process (a cudaDeviceReset of that device would make it stale).
fadam_status arena_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(FADAM_ELIMIT, "device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_arena_mutex);
  if (!g_arena_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_arena);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_arena)");
    g_arena_ptr[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_arena_ptr[dev]);
  return FADAM_OK;
}

}  // namespace

extern "C" fadam_status fadam_step_noalloc(const fadam_tensor* tensors, int64_t n_tensors,
                                           const fadam_group* groups, int32_t n_groups,
                                           int32_t p_dtype, int32_t g_dtype, int32_t out_dtype,
                                           uint32_t flags, int32_t* noop_dev,
                                           fadam_stream stream) {
  t_last_error.clear();
  const Dtypes d = make_dtypes(p_dtype, g_dtype, out_dtype, flags);
  if (flags & FADAM_SCALED_STATES)
    return fail(FADAM_EINVAL, "scaled states need a plan (fadam_plan_set_state_scales)");
  if ((flags & FADAM_CHECK_FINITE) && !noop_dev)
    return fail(FADAM_EINVAL, "FADAM_CHECK_FINITE needs a noop_dev flag to write");
  if (noop_dev && reinterpret_cast<uintptr_t>(noop_dev) % 4)
    return fail(FADAM_EALIGN, "noop_dev is not 4-byte aligned");
  // each call uploads its work list from host vectors that are gone when
  // it returns, so a captured call would leave a graph replaying garbage:
  // refuse a capturing stream (the implicit-capture error of the legacy
  // stream while another stream captures counts as capturing)
  {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap);
    if (ce == cudaErrorStreamCaptureImplicit || (ce == cudaSuccess && cap != cudaStreamCaptureStatusNone)) {
      cudaGetLastError();
      return fail(FADAM_EINVAL, "fadam_step_noalloc is not for stream capture (the stream is "
                                "capturing); use fadam_plan_create/fadam_step in a graph");
    }
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
  }
  HostPlan hp;
  fadam_status st = prepare(tensors, n_tensors, groups, n_groups, d, flags, true, kNoAllocMaxChunks,
                            hp);
  if (st) return st;
  if (static_cast<int64_t>(hp.items.size()) > kNoAllocMaxItems)
    return fail(FADAM_ELIMIT,
                "fadam_step_noalloc: the shard packs into %zu work items, more than the %lld its "
                "static device array holds; use fadam_plan_create/fadam_step",
                hp.items.size(), (long long)kNoAllocMaxItems);
  if (hp.grid > kNoAllocMaxCtas)
    return fail(FADAM_ELIMIT, "fadam_step_noalloc: grid of %d CTAs exceeds %d", hp.grid,
                kNoAllocMaxCtas);
  if (!needs_launch(hp)) return FADAM_OK;
  DeviceGuard guard(hp.device);
  if (guard.err != cudaSuccess) return cuda_fail(guard.err, "cudaSetDevice");
  unsigned char* arena = nullptr;
  st = arena_address(hp.device, &arena);
  if (st) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Item* items = reinterpret_cast<Item*>(arena + kArenaItemsOff);
  Chunk* chunks = reinterpret_cast<Chunk*>(arena + kArenaChunksOff);
  int32_t* cta = reinterpret_cast<int32_t*>(arena + kArenaCtaOff);
  KScratch* scratch = reinterpret_cast<KScratch*>(arena + kArenaScratchOff);
  cudaError_t e = cudaSuccess;
  if (!hp.items.empty())
    e = cudaMemcpyAsync(items, hp.items.data(), hp.items.size() * sizeof(Item),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !hp.chunks.empty())
    e = cudaMemcpyAsync(chunks, hp.chunks.data(), hp.chunks.size() * sizeof(Chunk),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cta, hp.cta_begin.data(), hp.cta_begin.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  // the counters and the status word must start at zero on every call
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(KScratch), s);
  if (e != cudaSuccess) return cuda_fail(e, "fadam_step_noalloc upload");
  KParams kp;
  fill_params(kp, items, cta, chunks, static_cast<int32_t>(hp.chunks.size()), noop_dev, scratch,
              groups, n_groups, flags | hp.shape);
  // the memo is shared by every call: its entries are keyed by betas and
  // step, so any entry that matches holds the corrections this call needs
  kp.memo = reinterpret_cast<BcMemo*>(arena + kArenaMemoOff);
  return launch(hp.kernel, hp.smem, kp, hp.grid, (flags & FADAM_CHECK_FINITE) != 0, s);
}
