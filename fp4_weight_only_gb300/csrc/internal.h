// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace petit {

constexpr uint32_t kStatusTimeout = 1u;  // bits in the workspace status word
constexpr uint32_t kStatusBounds = 2u;   // (bounds-checking build only)

// Workspace: [0, 256) status word and reserved; [256, 4352) split-tile
// arrival counters (u32), one per CTA index -- a split tile counts on the
// counter of its first contributing CTA, and a CTA is the first contributor
// of at most one split tile (the last tile of its range); then FP32 split-K
// partial slots, two per CTA.  The counter region has the same place and
// size for every problem, so no call's partials ever land on another
// call's counters and a workspace can be shared by problems of any shape.
constexpr size_t kWsHeaderBytes = 256;
// Largest grid whose stream-K ranges are given as an explicit table (a
// GB300 has 152 SMs); larger grids split the units evenly.
constexpr int kMaxBoundCtas = 160;
constexpr int kMaxCtas = 1024;
constexpr size_t kWsCountersBytes = sizeof(uint32_t) * kMaxCtas;

struct WsLayout {
  size_t counters_off;
  size_t partials_off;
  size_t total;
};

// A launch computes one GEMM or a group of GEMMs that share n and k (the
// experts of an MoE layer): group g multiplies activation rows
// [row_off[g], row_off[g+1]) by its own weights.  Tiles are numbered group by
// group (tile_base[g] is group g's first), weight-tile-major within a group.
constexpr int kMaxGroups = 64;

struct GemmPlan {
  int fmt;
  int bn;          // activation rows per tile (MMA N)
  int ku;          // 128-k chunks per pipeline unit (1 or 2)
  // CTA pairs: two CTAs of a cluster per work range, on a pair of adjacent
  // 128-row weight tiles (cta_group::2 MMAs); work tiles are then 256
  // weight rows and num_ctas counts work ranges (pairs)
  bool pair;
  int n_tiles;     // work tiles along n
  int k_stages;    // 128-k chunks per tile row
  int64_t units;   // tiles * k_stages / ku
  int num_ctas;    // work ranges (CTAs, or CTA pairs)
  // stream-K ranges: CTA c covers units [bound[c], bound[c+1]) when
  // use_bounds, else an even split
  bool use_bounds;
  int32_t bound[kMaxBoundCtas + 1];
  bool weights_reused;   // some group has several activation tiles
  int num_groups;
  int32_t row_off[kMaxGroups + 1];
  int32_t tile_base[kMaxGroups + 1];
  WsLayout ws;
};

// pair_cap: CTA pairs that can be resident at once (pair_capacity()), 0 to
// plan without CTA pairs
GemmPlan plan_gemm(int64_t m, int64_t n, int64_t k, int fmt, int num_sms, int pair_cap);
// Process-wide forced tile shape for the planner (tuning and tests): bn in
// {16, 32, 64, 128, 256}, ku in {1, 2} (2 only for bn <= 64); (0, 0) clears.
// Returns false for any other pair.
bool set_tile_override(int bn, int ku);
int tile_override();   // bn | ku << 16, or 0
// Whether this library is the bounds-checking build; in it, the extents the
// GEMM kernel's checks use (weight bytes per group, elements of C) may be
// lowered for tests (negative: the true extent).  Returns false in the
// normal build.
bool bounds_checking();
bool set_check_limits(int64_t weight_bytes, int64_t c_elems);
// row_off: num_groups + 1 non-decreasing offsets starting at 0
GemmPlan plan_grouped(const int64_t* row_off, int num_groups, int64_t n, int64_t k, int fmt,
                      int num_sms, int pair_cap);
// Resident CTA pairs of the pair kernels on the current device (0 if none).
int pair_capacity();
// 0: CTA pairs where the planner expects them to pay, 1: never, 2: wherever
// they apply (tests and tuning).  Returns false for any other value.
bool set_pair_mode(int mode);

struct GemmArgs {
  const void* A;
  const uint8_t* rep;   // repacked codes + scales
  void* C;
  int64_t m, n, k;
  float alpha;
  uint8_t* workspace;
  uint64_t timeout_ns;
  // if set, the epilogue factor is alpha_scale * (*alpha_dev), read on the
  // device after the preceding kernel on the stream has completed
  const float* alpha_dev = nullptr;
  float alpha_scale = 1.0f;
  // groups: bytes between consecutive groups' repacked weights, and each
  // group's epilogue factor (host array of num_groups; null: alpha for all)
  int64_t rep_stride = 0;
  const float* group_alpha = nullptr;
  int device = 0;   // the current device (the caller has looked it up)
};

cudaError_t launch_gemm(const GemmPlan& plan, const GemmArgs& args, const CUtensorMap& tmap_a,
                        cudaStream_t stream);

cudaError_t launch_absmax(const void* x, int64_t count, float* out, cudaStream_t stream);
cudaError_t launch_quantize(int fmt, const void* W, float g, uint8_t* wp, uint8_t* sp,
                            int64_t n, int64_t k, cudaStream_t stream);
cudaError_t launch_repack(int fmt, const uint8_t* wp, const uint8_t* sp, uint8_t* out,
                          int64_t n, int64_t k, cudaStream_t stream);
cudaError_t launch_dequant(int fmt, const uint8_t* rep, void* out, int64_t n, int64_t k,
                           cudaStream_t stream);
cudaError_t launch_selftest_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace petit
