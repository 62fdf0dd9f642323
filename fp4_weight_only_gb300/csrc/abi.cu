// C ABI: argument validation, problem planning, tensor-map encoding and
// kernel dispatch.  Validation always comes first and never touches the GPU,
// so a rejected call enqueues nothing.
#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/petit.h"
#include "fp4_layout.cuh"
#include "internal.h"

namespace {

using petit::kMXFP4;
using petit::kNVFP4;
using petit::kNVFP4F16;

constexpr int64_t kMaxDim = int64_t(1) << 24;
constexpr uint64_t kGemmTimeoutNs = 2000000000ull;  // no legitimate wait lasts 2 s
// the kernel counts a CTA's pipeline units in 32 bits
constexpr int64_t kMaxUnits = int64_t(1) << 31;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device facts, probed once.  state: 0 not probed, 1 usable (CC 10.3),
// 2 another architecture; num_sms is written before state is published
// (release), so the common path is one acquire load and no lock.
struct DevInfo {
  std::atomic<int> state{0};
  int num_sms = 0;
  int pair_cap = 0;   // resident CTA pairs of the pair kernels
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;   // only for the first probe of a device
DevInfo g_dev[kMaxDevices];

// Current device (one cudaGetDevice), its SM count, how many CTA pairs of
// the pair kernels it holds at once, and whether it is a compute-capability
// 10.3 part (the only code this library contains is sm_103a).
petit_status_t current_device(int* sms, int* dev_out = nullptr, int* pair_cap = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PETIT_ERR_CUDA;
  }
  DevInfo& d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
      int major = 0, minor = 0, n = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return PETIT_ERR_CUDA;
      }
      d.num_sms = n;
      st = (major == 10 && minor == 3) ? 1 : 2;
      d.pair_cap = st == 1 ? petit::pair_capacity() : 0;
      d.state.store(st, std::memory_order_release);
    }
  }
  if (sms) *sms = d.num_sms;
  if (dev_out) *dev_out = dev;
  if (pair_cap) *pair_cap = d.pair_cap;
  return st == 1 ? PETIT_OK : PETIT_ERR_ARCH;
}

petit_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? PETIT_OK : PETIT_ERR_CUDA; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// A [m][k] BF16 viewed as [k/64 slabs][m rows][64 k]: one box brings 2*ku
// slabs of 64 k for bn rows (128-byte swizzle, zero fill for rows >= m), i.e.
// a whole pipeline unit's activations in one request.
petit_status_t encode_a_map(CUtensorMap* map, const void* A, int64_t m, int64_t k, int bn,
                            int ku, bool f16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PETIT_ERR_CUDA;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(k / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(bn), static_cast<cuuint32_t>(2 * ku)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(A), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PETIT_OK : PETIT_ERR_CUDA;
}

// Activation tensor maps of recent calls, per host thread (no locking):
// serving loops call the GEMM with the same activation buffers and shapes
// over and over, and encoding a map costs more than the rest of the call.
// The key is everything the map encodes.
struct MapKey {
  const void* A;
  int64_t m, k;
  int bn, ku, f16, dev;
};

petit_status_t cached_a_map(CUtensorMap* map, const void* A, int64_t m, int64_t k, int bn, int ku,
                            bool f16, int dev) {
  constexpr int kSlots = 8;
  thread_local MapKey keys[kSlots];
  thread_local CUtensorMap maps[kSlots];
  thread_local int used = 0, next = 0;
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.A = A;
  key.m = m;
  key.k = k;
  key.bn = bn;
  key.ku = ku;
  key.f16 = f16 ? 1 : 0;
  key.dev = dev;
  for (int i = 0; i < used; ++i) {
    if (std::memcmp(&keys[i], &key, sizeof(key)) == 0) {
      *map = maps[i];
      return PETIT_OK;
    }
  }
  std::memset(map, 0, sizeof(*map));
  if (petit_status_t st = encode_a_map(map, A, m, k, bn, ku, f16)) return st;
  keys[next] = key;
  maps[next] = *map;
  next = (next + 1) % kSlots;
  if (used < kSlots) ++used;
  return PETIT_OK;
}

petit_status_t check_tiled_shape(int64_t n, int64_t k) {
  if (n < petit::kTileN || k < petit::kStageK || n % petit::kTileN || k % petit::kStageK ||
      n > kMaxDim || k > kMaxDim)
    return PETIT_ERR_UNSUPPORTED_SHAPE;
  return PETIT_OK;
}

petit_status_t gemm_common(int fmt, const void* A, const uint8_t* rep, float alpha, void* C,
                           int64_t m, int64_t n, int64_t k, void* ws, size_t ws_bytes,
                           petit_stream_t stream, const float* alpha_dev = nullptr) {
  if (!A || !rep || !C || m < 1) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (m > kMaxDim) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(rep) || !aligned16(C)) return PETIT_ERR_MISALIGNED;
  if (!ws) return PETIT_ERR_WORKSPACE;
  if (!aligned16(ws)) return PETIT_ERR_MISALIGNED;
  int sms = 0, dev = 0;
  int pair_cap = 0;
  if (petit_status_t st = current_device(&sms, &dev, &pair_cap)) return st;
  const petit::GemmPlan plan = petit::plan_gemm(m, n, k, fmt, sms, pair_cap);
  if (plan.units >= kMaxUnits) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < plan.ws.total) return PETIT_ERR_WORKSPACE;
  CUtensorMap map;
  // (CTA pairs: each CTA's activation box holds half of a tile's rows)
  if (petit_status_t st = cached_a_map(&map, A, m, k, plan.pair ? plan.bn / 2 : plan.bn, plan.ku,
                                       fmt == kNVFP4F16, dev))
    return st;
  petit::GemmArgs args{A, rep, C, m, n, k, alpha, static_cast<uint8_t*>(ws), kGemmTimeoutNs};
  args.device = dev;
  if (alpha_dev) {
    args.alpha_dev = alpha_dev;
    args.alpha_scale = alpha;
  }
  return from_cuda(petit::launch_gemm(plan, args, map, reinterpret_cast<cudaStream_t>(stream)));
}

// Checks expert offsets: 1 <= E <= kMaxGroups, off[0] == 0, non-decreasing,
// total rows <= kMaxDim.
petit_status_t check_offsets(const int64_t* off, int64_t num_experts) {
  if (!off || num_experts < 1) return PETIT_ERR_INVALID_ARG;
  if (num_experts > petit::kMaxGroups) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (off[0] != 0) return PETIT_ERR_INVALID_ARG;
  for (int64_t e = 0; e < num_experts; ++e)
    if (off[e + 1] < off[e]) return PETIT_ERR_INVALID_ARG;
  if (off[num_experts] > kMaxDim) return PETIT_ERR_UNSUPPORTED_SHAPE;
  return PETIT_OK;
}

petit_status_t moe_common(int fmt, const void* A, const uint8_t* rep, const float* gscales,
                          const int64_t* off, int64_t num_experts, void* C, int64_t n, int64_t k,
                          void* ws, size_t ws_bytes, petit_stream_t stream) {
  if (petit_status_t st = check_offsets(off, num_experts)) return st;
  if (off[num_experts] == 0) return PETIT_OK;   // no routed tokens: nothing to compute
  if (!A || !rep || !C) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (!aligned16(A) || !aligned16(rep) || !aligned16(C)) return PETIT_ERR_MISALIGNED;
  float alphas[petit::kMaxGroups];
  for (int64_t e = 0; e < num_experts; ++e) {
    const float g = gscales ? gscales[e] : 1.0f;
    if (!(g > 0.0f) || g > 1.0e36f) return PETIT_ERR_INVALID_ARG;
    // NVFP4's register decode yields Wq * 2^-8; the epilogue restores it
    alphas[e] = fmt == kNVFP4 ? g * 256.0f : 1.0f;
  }
  const int64_t rows = off[num_experts];
  if (!ws) return PETIT_ERR_WORKSPACE;
  if (!aligned16(ws)) return PETIT_ERR_MISALIGNED;
  int sms = 0, dev = 0;
  int pair_cap = 0;
  if (petit_status_t st = current_device(&sms, &dev, &pair_cap)) return st;
  const petit::GemmPlan plan =
      petit::plan_grouped(off, static_cast<int>(num_experts), n, k, fmt, sms, pair_cap);
  if (plan.units >= kMaxUnits) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < plan.ws.total) return PETIT_ERR_WORKSPACE;
  CUtensorMap map;
  if (petit_status_t st = cached_a_map(&map, A, rows, k, plan.pair ? plan.bn / 2 : plan.bn,
                                       plan.ku, false, dev))
    return st;
  petit::GemmArgs args{A, rep, C, rows, n, k, alphas[0], static_cast<uint8_t*>(ws), kGemmTimeoutNs};
  args.device = dev;
  args.rep_stride = static_cast<int64_t>(petit_repacked_bytes(n, k, fmt));
  args.group_alpha = alphas;
  return from_cuda(petit::launch_gemm(plan, args, map, reinterpret_cast<cudaStream_t>(stream)));
}

// Arguments of the plan queries that do not depend on the problem.
petit_status_t check_plan_args(int num_sms, int pair_cap, const petit_plan_info_t* info) {
  if (!info || num_sms < 1 || num_sms > petit::kMaxCtas || pair_cap < 0 ||
      pair_cap > petit::kMaxBoundCtas)
    return PETIT_ERR_INVALID_ARG;
  return PETIT_OK;
}

// A plan as the public struct, and its ranges: the first unit of range c is
// the kernel's own cta_lo(c) (explicit bounds, else the even split
// c * (U / P) + c * (U % P) / P).
petit_status_t describe_plan(const petit::GemmPlan& pl, petit_plan_info_t* info,
                             int64_t* starts, int64_t max_ranges) {
  if (pl.units >= kMaxUnits) return PETIT_ERR_UNSUPPORTED_SHAPE;
  std::memset(info, 0, sizeof(*info));
  info->bn = pl.bn;
  info->ku = pl.ku;
  info->cta_pairs = pl.pair ? 1 : 0;
  info->num_ranges = pl.num_ctas;
  info->num_ctas = pl.num_ctas * (pl.pair ? 2 : 1);
  info->units_per_tile = pl.k_stages / pl.ku;
  info->num_tiles = info->units_per_tile > 0 ? pl.units / info->units_per_tile : 0;
  info->units = pl.units;
  info->workspace_bytes = pl.ws.total;
  if (!starts) return PETIT_OK;
  const int64_t P = pl.num_ctas;
  if (max_ranges < P + 1) return PETIT_ERR_INVALID_ARG;
  const int64_t q = pl.units / P, r = pl.units % P;
  for (int64_t c = 0; c <= P; ++c)
    starts[c] = c == P ? pl.units : pl.use_bounds ? pl.bound[c] : c * q + (c * r) / P;
  return PETIT_OK;
}

}  // namespace

extern "C" {

int petit_layout_version(void) { return petit::kLayoutVersion; }

const char* petit_status_string(petit_status_t s) {
  switch (s) {
    case PETIT_OK: return "ok";
    case PETIT_ERR_INVALID_ARG: return "invalid argument";
    case PETIT_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case PETIT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case PETIT_ERR_WORKSPACE: return "workspace missing or too small";
    case PETIT_ERR_ARCH: return "device is not sm_103 (GB300)";
    case PETIT_ERR_CUDA: return "CUDA runtime error";
    case PETIT_ERR_TIMEOUT: return "device-side wait timed out";
    case PETIT_ERR_BOUNDS: return "device-side index check failed";
  }
  return "unknown status";
}

size_t petit_repacked_bytes(int64_t n, int64_t k, int fmt) {
  if (n < 0 || k < 0) return 0;
  const size_t nk = static_cast<size_t>(n) * static_cast<size_t>(k);
  if (fmt == PETIT_FMT_NVFP4 || fmt == PETIT_FMT_NVFP4_F16) return nk / 2 + nk / 16;
  // MXFP4 chunks (128 x 128) carry a 16-byte flag field: nk / 1024 bytes
  if (fmt == PETIT_FMT_MXFP4) return nk / 2 + nk / 32 + nk / 1024;
  return 0;
}

size_t petit_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int fmt) {
  if (m < 1 || m > kMaxDim || check_tiled_shape(n, k) != PETIT_OK) return 0;
  if (fmt != PETIT_FMT_NVFP4 && fmt != PETIT_FMT_MXFP4 && fmt != PETIT_FMT_NVFP4_F16) return 0;
  int sms = 0;
  int pair_cap = 0;
  if (current_device(&sms, nullptr, &pair_cap) != PETIT_OK) return 0;
  return petit::plan_gemm(m, n, k, fmt, sms, pair_cap).ws.total;
}

size_t petit_moe_workspace_bytes(const int64_t* expert_offsets, int64_t num_experts, int64_t n,
                                 int64_t k, int fmt) {
  if (check_offsets(expert_offsets, num_experts) != PETIT_OK || check_tiled_shape(n, k) != PETIT_OK)
    return 0;
  if (fmt != PETIT_FMT_NVFP4 && fmt != PETIT_FMT_MXFP4) return 0;
  int sms = 0;
  int pair_cap = 0;
  if (current_device(&sms, nullptr, &pair_cap) != PETIT_OK) return 0;
  return petit::plan_grouped(expert_offsets, static_cast<int>(num_experts), n, k, fmt, sms,
                             pair_cap)
      .ws.total;
}

petit_status_t petit_moe_gemm_bf16_mxfp4(const void* A, const uint8_t* rep,
                                         const int64_t* expert_offsets, int64_t num_experts,
                                         void* C, int64_t n, int64_t k, void* workspace,
                                         size_t workspace_bytes, petit_stream_t stream) {
  return moe_common(kMXFP4, A, rep, nullptr, expert_offsets, num_experts, C, n, k, workspace,
                    workspace_bytes, stream);
}

petit_status_t petit_moe_gemm_bf16_nvfp4(const void* A, const uint8_t* rep,
                                         const float* global_scales, const int64_t* expert_offsets,
                                         int64_t num_experts, void* C, int64_t n, int64_t k,
                                         void* workspace, size_t workspace_bytes,
                                         petit_stream_t stream) {
  if (!global_scales) return PETIT_ERR_INVALID_ARG;
  return moe_common(kNVFP4, A, rep, global_scales, expert_offsets, num_experts, C, n, k, workspace,
                    workspace_bytes, stream);
}

petit_status_t petit_absmax_bf16(const void* x, int64_t count, float* amax_out,
                                 petit_stream_t stream) {
  if (!x || !amax_out || count < 1) return PETIT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(amax_out) & 3u))
    return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(petit::launch_absmax(x, count, amax_out, reinterpret_cast<cudaStream_t>(stream)));
}

float petit_nvfp4_global_scale(float amax) { return amax / (6.0f * 448.0f); }

static petit_status_t quantize_common(int fmt, const void* W, float g, uint8_t* wp, uint8_t* sp,
                                      int64_t n, int64_t k, petit_stream_t stream) {
  if (!W || !wp || !sp || n < 1 || k < 1) return PETIT_ERR_INVALID_ARG;
  const int64_t blk = fmt == PETIT_FMT_NVFP4 ? 16 : 32;
  if (k % blk || n > kMaxDim || k > kMaxDim) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W) || !aligned16(wp) || !aligned16(sp)) return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(
      petit::launch_quantize(fmt, W, g, wp, sp, n, k, reinterpret_cast<cudaStream_t>(stream)));
}

petit_status_t petit_quantize_nvfp4(const void* W, float global_scale, uint8_t* w_packed,
                                    uint8_t* s_e4m3, int64_t n, int64_t k,
                                    petit_stream_t stream) {
  if (!(global_scale > 0.0f) || global_scale > 3.0e38f) return PETIT_ERR_INVALID_ARG;
  return quantize_common(kNVFP4, W, global_scale, w_packed, s_e4m3, n, k, stream);
}

petit_status_t petit_quantize_mxfp4(const void* W, uint8_t* w_packed, uint8_t* s_e8m0, int64_t n,
                                    int64_t k, petit_stream_t stream) {
  return quantize_common(kMXFP4, W, 1.0f, w_packed, s_e8m0, n, k, stream);
}

static petit_status_t repack_common(int fmt, const uint8_t* wp, const uint8_t* sp, uint8_t* out,
                                    int64_t n, int64_t k, petit_stream_t stream) {
  if (!wp || !sp || !out) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (!aligned16(wp) || !aligned16(sp) || !aligned16(out)) return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(
      petit::launch_repack(fmt, wp, sp, out, n, k, reinterpret_cast<cudaStream_t>(stream)));
}

petit_status_t petit_repack_nvfp4(const uint8_t* w_packed, const uint8_t* s_e4m3, uint8_t* rep_out,
                                  int64_t n, int64_t k, petit_stream_t stream) {
  return repack_common(kNVFP4, w_packed, s_e4m3, rep_out, n, k, stream);
}

petit_status_t petit_repack_nvfp4_f16(const uint8_t* w_packed, const uint8_t* s_e4m3,
                                      uint8_t* rep_out, int64_t n, int64_t k,
                                      petit_stream_t stream) {
  return repack_common(kNVFP4F16, w_packed, s_e4m3, rep_out, n, k, stream);
}

petit_status_t petit_repack_mxfp4(const uint8_t* w_packed, const uint8_t* s_e8m0, uint8_t* rep_out,
                                  int64_t n, int64_t k, petit_stream_t stream) {
  return repack_common(kMXFP4, w_packed, s_e8m0, rep_out, n, k, stream);
}

petit_status_t petit_dequant_bf16(const uint8_t* rep, int fmt, void* W_out, int64_t n, int64_t k,
                                  petit_stream_t stream) {
  if (!rep || !W_out) return PETIT_ERR_INVALID_ARG;
  if (fmt != PETIT_FMT_NVFP4 && fmt != PETIT_FMT_MXFP4) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (!aligned16(rep) || !aligned16(W_out)) return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(
      petit::launch_dequant(fmt, rep, W_out, n, k, reinterpret_cast<cudaStream_t>(stream)));
}

petit_status_t petit_dequant_f16(const uint8_t* rep, void* W_out, int64_t n, int64_t k,
                                 petit_stream_t stream) {
  if (!rep || !W_out) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (!aligned16(rep) || !aligned16(W_out)) return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(petit::launch_dequant(kNVFP4F16, rep, W_out, n, k,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

petit_status_t petit_gemm_f16_nvfp4(const void* A, const uint8_t* rep, float global_scale, void* C,
                                    int64_t m, int64_t n, int64_t k, void* workspace,
                                    size_t workspace_bytes, petit_stream_t stream) {
  if (!(global_scale > 0.0f) || global_scale > 1.0e36f) return PETIT_ERR_INVALID_ARG;
  // the FP16 register decode yields Wq * 2^-7; the epilogue restores it with g
  return gemm_common(kNVFP4F16, A, rep, global_scale * 128.0f, C, m, n, k, workspace,
                     workspace_bytes, stream);
}

petit_status_t petit_gemm_bf16_nvfp4(const void* A, const uint8_t* rep, float global_scale,
                                     void* C, int64_t m, int64_t n, int64_t k, void* workspace,
                                     size_t workspace_bytes, petit_stream_t stream) {
  if (!(global_scale > 0.0f) || global_scale > 1.0e36f) return PETIT_ERR_INVALID_ARG;
  // the register decode yields Wq * 2^-8; the epilogue restores it with g
  return gemm_common(kNVFP4, A, rep, global_scale * 256.0f, C, m, n, k, workspace,
                     workspace_bytes, stream);
}

petit_status_t petit_gemm_bf16_nvfp4_dscale(const void* A, const uint8_t* rep,
                                            const float* global_scale_dev, void* C, int64_t m,
                                            int64_t n, int64_t k, void* workspace,
                                            size_t workspace_bytes, petit_stream_t stream) {
  if (!global_scale_dev || reinterpret_cast<uintptr_t>(global_scale_dev) % 4 != 0)
    return PETIT_ERR_INVALID_ARG;
  return gemm_common(kNVFP4, A, rep, 256.0f, C, m, n, k, workspace, workspace_bytes, stream,
                     global_scale_dev);
}

petit_status_t petit_gemm_bf16_mxfp4(const void* A, const uint8_t* rep, void* C, int64_t m,
                                     int64_t n, int64_t k, void* workspace,
                                     size_t workspace_bytes, petit_stream_t stream) {
  return gemm_common(kMXFP4, A, rep, 1.0f, C, m, n, k, workspace, workspace_bytes, stream);
}

petit_status_t petit_set_tile_config(int bn, int ku) {
  return petit::set_tile_override(bn, ku) ? PETIT_OK : PETIT_ERR_INVALID_ARG;
}

petit_status_t petit_set_pair_mode(int mode) {
  return petit::set_pair_mode(mode) ? PETIT_OK : PETIT_ERR_INVALID_ARG;
}

petit_status_t petit_plan_gemm(int64_t m, int64_t n, int64_t k, int fmt, int num_sms,
                               int pair_capacity, petit_plan_info_t* info,
                               int64_t* range_starts, int64_t max_ranges) {
  if (petit_status_t st = check_plan_args(num_sms, pair_capacity, info)) return st;
  if (m < 1) return PETIT_ERR_INVALID_ARG;
  if (fmt != PETIT_FMT_NVFP4 && fmt != PETIT_FMT_MXFP4 && fmt != PETIT_FMT_NVFP4_F16)
    return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (m > kMaxDim) return PETIT_ERR_UNSUPPORTED_SHAPE;
  return describe_plan(petit::plan_gemm(m, n, k, fmt, num_sms, pair_capacity), info,
                       range_starts, max_ranges);
}

petit_status_t petit_plan_moe(const int64_t* expert_offsets, int64_t num_experts, int64_t n,
                              int64_t k, int fmt, int num_sms, int pair_capacity,
                              petit_plan_info_t* info, int64_t* range_starts,
                              int64_t max_ranges) {
  if (petit_status_t st = check_plan_args(num_sms, pair_capacity, info)) return st;
  if (fmt != PETIT_FMT_NVFP4 && fmt != PETIT_FMT_MXFP4) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_offsets(expert_offsets, num_experts)) return st;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (expert_offsets[num_experts] == 0) {   // the GEMM launches nothing
    std::memset(info, 0, sizeof(*info));
    return PETIT_OK;
  }
  return describe_plan(petit::plan_grouped(expert_offsets, static_cast<int>(num_experts), n, k,
                                           fmt, num_sms, pair_capacity),
                       info, range_starts, max_ranges);
}

petit_status_t petit_device_limits(int* num_sms, int* pair_capacity) {
  if (!num_sms || !pair_capacity) return PETIT_ERR_INVALID_ARG;
  int sms = 0, pc = 0;
  if (petit_status_t st = current_device(&sms, nullptr, &pc)) return st;
  *num_sms = sms;
  *pair_capacity = pc;
  return PETIT_OK;
}

int petit_bounds_checking(void) { return petit::bounds_checking() ? 1 : 0; }

petit_status_t petit_check_set_limits(int64_t weight_bytes, int64_t c_elems) {
  return petit::set_check_limits(weight_bytes, c_elems) ? PETIT_OK : PETIT_ERR_INVALID_ARG;
}

petit_status_t petit_get_device_status(void* workspace, size_t workspace_bytes,
                                       petit_stream_t stream) {
  if (!workspace || workspace_bytes < petit::kWsHeaderBytes) return PETIT_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return PETIT_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PETIT_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PETIT_ERR_CUDA;
  if (word == 0) return PETIT_OK;
  // A kernel that stopped early may have left split-tile arrival counters
  // raised (CTAs that had arrived before the abort); clear them with the
  // status word so the next call on this workspace starts from zero.
  const size_t counters_end = petit::kWsHeaderBytes + petit::kWsCountersBytes;
  const size_t clear = workspace_bytes >= counters_end ? counters_end : sizeof(word);
  if (cudaMemsetAsync(workspace, 0, clear, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return PETIT_ERR_CUDA;
  if (word & petit::kStatusBounds) return PETIT_ERR_BOUNDS;
  return (word & petit::kStatusTimeout) ? PETIT_ERR_TIMEOUT : PETIT_ERR_CUDA;
}

petit_status_t petit_selftest_timeout(void* workspace, size_t workspace_bytes, uint32_t timeout_us,
                                      petit_stream_t stream) {
  if (!workspace || timeout_us < 1 || timeout_us > 1000000u) return PETIT_ERR_INVALID_ARG;
  if (workspace_bytes < petit::kWsHeaderBytes) return PETIT_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PETIT_ERR_MISALIGNED;
  if (petit_status_t st = current_device(nullptr)) return st;
  return from_cuda(petit::launch_selftest_timeout(static_cast<uint32_t*>(workspace),
                                                  uint64_t(timeout_us) * 1000ull,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// GEMM without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the GEMM:
// plug-ins whose host framework owns all device memory and forbids
// allocation inside their enqueue call, and latency-critical serving loops
// where cudaMalloc's implicit device synchronisation is unacceptable.
// For them the split-K scratch (status word, arrival counters, FP32 partial
// sums) lives in a fixed array in this library's device image instead of a
// caller buffer.
namespace {

// Size of the built-in scratch.  Every GPU that loads the library keeps this
// much device memory until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" petit_status_t petit_gemm_bf16_nvfp4_noalloc(const void* A, const uint8_t* rep,
                                                        float global_scale, void* C, int64_t m,
                                                        int64_t n, int64_t k,
                                                        petit_stream_t stream) {
  if (!(global_scale > 0.0f) || global_scale > 1.0e36f) return PETIT_ERR_INVALID_ARG;
  if (!A || !rep || !C || m < 1) return PETIT_ERR_INVALID_ARG;
  if (petit_status_t st = check_tiled_shape(n, k)) return st;
  if (m > kMaxDim) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(rep) || !aligned16(C)) return PETIT_ERR_MISALIGNED;
  int sms = 0;
  int pair_cap = 0;
  if (petit_status_t st = current_device(&sms, nullptr, &pair_cap)) return st;
  const petit::GemmPlan plan = petit::plan_gemm(m, n, k, kNVFP4, sms, pair_cap);
  if (plan.units >= kMaxUnits) return PETIT_ERR_UNSUPPORTED_SHAPE;
  if (plan.ws.total > kNoAllocScratchBytes) return PETIT_ERR_WORKSPACE;  // problem too large
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PETIT_ERR_CUDA;
  void* scratch = nullptr;
  {
    // first call on a device (with that device current): look up the
    // array's device address -- in host code its name is only a host-side
    // stand-in, never a device address.  The address is kept for the life of
    // the process; cudaDeviceReset unloads the module and makes it stale, so
    // this entry point must not be used after a reset of that device.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return PETIT_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // every check that can fail comes before the first enqueue
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  if (petit_status_t st =
          encode_a_map(&map, A, m, k, plan.pair ? plan.bn / 2 : plan.bn, plan.ku))
    return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word and the arrival counters must start at zero; the array
  // keeps whatever the previous call left in it
  if (cudaMemsetAsync(scratch, 0, plan.ws.partials_off, s) != cudaSuccess) return PETIT_ERR_CUDA;
  petit::GemmArgs args{A, rep, C, m, n, k, global_scale * 256.0f, static_cast<uint8_t*>(scratch),
                       kGemmTimeoutNs};
  args.device = dev;
  return from_cuda(petit::launch_gemm(plan, args, map, s));
}
