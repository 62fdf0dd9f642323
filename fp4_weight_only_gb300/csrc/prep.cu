// Offline weight preparation: max-abs, NVFP4 / MXFP4 quantisation, the
// Marlin-style repack, the dequantisation test hook and the bounded-wait self
// test.  All memory-bound, one pass each.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fp4_layout.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace petit {
namespace {

constexpr int kThreads = 256;

// Blocks for a grid-stride kernel over `work` items: one item per thread, at
// most 32 blocks per SM of the current device (the kernels loop beyond that).
int grid_for(int64_t work, int per_block = kThreads) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    sms = 1;
  }
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > static_cast<int64_t>(sms) * 32) g = static_cast<int64_t>(sms) * 32;
  return static_cast<int>(g);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Nearest E2M1 code of y, ties to the even-mantissa neighbour, saturating at
// 6; magnitude 0 always gives code 0 (no negative zero).  The grid is
// {0, .5, 1, 1.5, 2, 3, 4, 6} ("FP4 GEMM on Rubin/Blackwell with CUTLASS",
// section 2.1); the thresholds are the midpoints, with '>' where the lower
// neighbour is even and '>=' where the upper one is.
__device__ __forceinline__ uint32_t e2m1_nearest(float y) {
  const float a = fabsf(y);
  const uint32_t i = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return i | ((y < 0.0f && i != 0u) ? 8u : 0u);
}

// FP32 -> E4M3FN, round to nearest even, saturating to +-448 (hardware cvt;
// both halves get the same value so the byte order does not matter).
__device__ __forceinline__ uint32_t f32_to_e4m3(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(t));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(b | (b << 8))));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// ------------------------------------------------------------------ max-abs
__global__ void absmax_kernel(const __nv_bfloat16* __restrict__ x, int64_t count,
                              unsigned int* __restrict__ out) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nvec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) ? count / 8 : 0;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  for (int64_t i = tid; i < nvec; i += stride) {
    float f[8];
    bf16x8_to_f32(xv[i], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
  for (int64_t i = nvec * 8 + tid; i < count; i += stride) m = fmaxf(m, fabsf(__bfloat162float(x[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));  // m >= 0: bits order as floats
}

// ---------------------------------------------------------------- quantise
// NVFP4: one thread per 16-element block.  Scale and division in FP32 with
// IEEE rounding (the precision the CPU oracle reproduces).
__global__ void quantize_nvfp4_kernel(const __nv_bfloat16* __restrict__ W, float g,
                                      uint8_t* __restrict__ wp, uint8_t* __restrict__ sp,
                                      int64_t nblocks) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float denom = 6.0f * g;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
       b += stride) {
    const uint4* src = reinterpret_cast<const uint4*>(W) + 2 * b;
    float x[16];
    float (&x0)[8] = *reinterpret_cast<float(*)[8]>(&x[0]);
    float (&x1)[8] = *reinterpret_cast<float(*)[8]>(&x[8]);
    bf16x8_to_f32(src[0], x0);
    bf16x8_to_f32(src[1], x1);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float t = fmaxf(amax, 1e-8f) / denom;
    uint32_t sc = f32_to_e4m3(t);
    if (sc == 0u) sc = 1u;                       // keep every scale positive
    const float d = e4m3_to_f32(sc) * g;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) lo |= e2m1_nearest(x[i] / d) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) hi |= e2m1_nearest(x[8 + i] / d) << (4 * i);
    reinterpret_cast<uint2*>(wp)[b] = make_uint2(lo, hi);
    sp[b] = static_cast<uint8_t>(sc);
  }
}

// MXFP4: one thread per 32-element block; scale 2^ceil(log2(max(amax,1e-8)/6)).
__global__ void quantize_mxfp4_kernel(const __nv_bfloat16* __restrict__ W,
                                      uint8_t* __restrict__ wp, uint8_t* __restrict__ sp,
                                      int64_t nblocks) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
       b += stride) {
    const uint4* src = reinterpret_cast<const uint4*>(W) + 4 * b;
    float x[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float (&xv)[8] = *reinterpret_cast<float(*)[8]>(&x[8 * v]);
      bf16x8_to_f32(src[v], xv);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float y = fmaxf(amax, 1e-8f) / 6.0f;    // a normal number, >= 1.6e-9
    const uint32_t bits = __float_as_uint(y);
    const int ef = static_cast<int>(bits >> 23);
    int e = (bits & 0x7FFFFFu) ? ef - 126 : ef - 127;  // exact ceil(log2 y)
    int c = e + 127;
    c = c < 0 ? 0 : (c > 254 ? 254 : c);
    e = c - 127;
    const float inv = (e < 127) ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23)
                                : __uint_as_float(0x00400000u);  // 2^-e, exact
    uint32_t q[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 32; ++i) q[i >> 3] |= e2m1_nearest(x[i] * inv) << (4 * (i & 7));
    reinterpret_cast<uint4*>(wp)[b] = make_uint4(q[0], q[1], q[2], q[3]);
    sp[b] = static_cast<uint8_t>(c);
  }
}

// ------------------------------------------------------------------- repack
// One CTA per (stage, tile) chunk: 128 rows x 64 bytes of packed codes are
// staged through shared memory so both the reads and the writes are
// contiguous; each 32-bit word's 8 codes are moved to their decode positions,
// and the chunk's scale bytes are appended after its codes.
template <int FMT>
__global__ void __launch_bounds__(kThreads) repack_kernel(const uint8_t* __restrict__ wp,
                                                          const uint8_t* __restrict__ sp,
                                                          uint8_t* __restrict__ out, int64_t k) {
  using T = FmtTraits<FMT>;
  const int64_t stages = k / kStageK;
  const int64_t s = blockIdx.x;
  const int64_t t = blockIdx.y;
  __shared__ uint4 tile[kTileN][kGroupsPerRow];
  const int64_t row_bytes = k / 2;
  for (int i = threadIdx.x; i < kTileN * kGroupsPerRow; i += kThreads) {
    const int r = i >> 2, g = i & 3;
    tile[r][g] = *reinterpret_cast<const uint4*>(wp + (t * kTileN + r) * row_bytes +
                                                 s * (kStageK / 2) + g * 16);
  }
  __syncthreads();
  uint8_t* dst = out + chunk_offset<FMT>(t, s, stages);
  for (int i = threadIdx.x; i < kTileN * kGroupsPerRow; i += kThreads) {
    const int g = i >> 7, r = i & 127;
    const uint4 in = tile[r][g];
    const uint32_t iw[4] = {in.x, in.y, in.z, in.w};
    uint32_t ow[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = (iw[w] >> (4 * j)) & 0xFu;
      ow[w] = FMT == kNVFP4F16 ? pack_word_f16(c) : pack_word(c);
    }
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(i) * 16) =
        make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
  // scales: half h of row r <- bytes [h * B, h * B + B) of the stage's bytes
  constexpr int B = T::kScaleBytesPerHalf;
  const int64_t srow_bytes = k / T::kBlock;
  uint8_t* sdst = dst + kWChunkBytes;
  for (int i = threadIdx.x; i < 2 * kTileN; i += kThreads) {
    const int h = i >> 7, r = i & 127;
    const uint8_t* src = sp + (t * kTileN + r) * srow_bytes + s * (2 * B) + h * B;
    if constexpr (B == 4) {
      *reinterpret_cast<uint32_t*>(sdst + i * 4) = *reinterpret_cast<const uint32_t*>(src);
    } else {
      *reinterpret_cast<uint16_t*>(sdst + i * 2) = *reinterpret_cast<const uint16_t*>(src);
    }
  }
  if constexpr (FMT == kMXFP4) {
    // the chunk's flag: every E8M0 code <= 128, so the decode may multiply
    // once by 2^(c - 1) (a BF16 number for those codes)
    bool small = true;
    for (int i = threadIdx.x; i < 2 * kTileN; i += kThreads) {
      const int h = i >> 7, r = i & 127;
      const uint8_t* src = sp + (t * kTileN + r) * srow_bytes + s * (2 * B) + h * B;
      small = small && src[0] <= 128 && src[1] <= 128;
    }
    small = __syncthreads_and(small) != 0;
    if (threadIdx.x == 0)
      *reinterpret_cast<uint4*>(sdst + T::kSChunkBytes) = make_uint4(small ? 1u : 0u, 0u, 0u, 0u);
  }
  // The GEMM reads its weights before its grid dependency wait, so it may
  // start (right after this kernel's CTAs exit) without the usual end-of-
  // kernel flush: make this thread's writes visible device-wide before it
  // exits, so a GEMM may directly follow the repack on the same stream.
  __threadfence();
}

// ------------------------------------------------------------- dequant hook
// One thread per (chunk, group, row): decodes 32 codes with the GEMM's decode
// and writes Wq = code * scale as BF16 [n][k] (FP16 for the FP16 layout).
template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ rep, uint16_t* __restrict__ out,
                               int64_t n, int64_t k) {
  using T = FmtTraits<FMT>;
  const int64_t stages = k / kStageK;
  const int64_t total = (n / kTileN) * stages * (kTileN * kGroupsPerRow);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t chunk = idx >> 9;
    const int within = static_cast<int>(idx & 511);
    const int g = within >> 7, r = within & 127, h = g >> 1;
    const int64_t t = chunk / stages, s = chunk % stages;
    const uint8_t* cbase = rep + chunk * T::kChunkBytes;
    const uint4 grp = *reinterpret_cast<const uint4*>(cbase + within * 16);
    uint32_t sc;
    if constexpr (FMT == kNVFP4 || FMT == kNVFP4F16) {
      sc = *reinterpret_cast<const uint16_t*>(cbase + kWChunkBytes + (h * 128 + r) * 4 + (g & 1) * 2);
    } else {
      sc = cbase[kWChunkBytes + (h * 128 + r) * 2 + (g & 1)];
    }
    uint32_t o[16];
    if constexpr (FMT == kMXFP4) {
      // the GEMM's two decodes, chosen by the chunk's flag
      if (cbase[kWChunkBytes + T::kSChunkBytes]) decode_group<FMT, true>(grp, sc, o);
      else decode_group<FMT>(grp, sc, o);
    } else {
      decode_group<FMT>(grp, sc, o);
    }
    if constexpr (FMT == kNVFP4) {
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = bmul2(o[j], kBf16x2_2p8);  // undo 2^-8, exact
    } else if constexpr (FMT == kNVFP4F16) {
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = hmul2(o[j], kF16x2_2p7);  // undo 2^-7, exact
    }
    uint4* dst = reinterpret_cast<uint4*>(out + (t * kTileN + r) * k + s * kStageK + g * 32);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
  }
}

// ---------------------------------------------------------------- self test
__global__ void selftest_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ alignas(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody arrives on `bar`: the bounded wait must give up and report
    if (!mbar_wait_bounded(smem_u32(&bar), 0, timeout_ns, nullptr)) atomicOr(status, kStatusTimeout);
  }
}

}  // namespace

cudaError_t launch_absmax(const void* x, int64_t count, float* out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  absmax_kernel<<<grid_for(count / 8 + 1), kThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), count, reinterpret_cast<unsigned int*>(out));
  return cudaGetLastError();
}

cudaError_t launch_quantize(int fmt, const void* W, float g, uint8_t* wp, uint8_t* sp, int64_t n,
                            int64_t k, cudaStream_t stream) {
  const auto* w = static_cast<const __nv_bfloat16*>(W);
  if (fmt == kNVFP4) {
    const int64_t nb = n * (k / 16);
    quantize_nvfp4_kernel<<<grid_for(nb), kThreads, 0, stream>>>(w, g, wp, sp, nb);
  } else {
    const int64_t nb = n * (k / 32);
    quantize_mxfp4_kernel<<<grid_for(nb), kThreads, 0, stream>>>(w, wp, sp, nb);
  }
  return cudaGetLastError();
}

cudaError_t launch_repack(int fmt, const uint8_t* wp, const uint8_t* sp, uint8_t* out,
                          int64_t n, int64_t k, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(k / kStageK), static_cast<unsigned>(n / kTileN));
  if (fmt == kNVFP4)
    repack_kernel<kNVFP4><<<grid, kThreads, 0, stream>>>(wp, sp, out, k);
  else if (fmt == kNVFP4F16)
    repack_kernel<kNVFP4F16><<<grid, kThreads, 0, stream>>>(wp, sp, out, k);
  else
    repack_kernel<kMXFP4><<<grid, kThreads, 0, stream>>>(wp, sp, out, k);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* rep, void* out, int64_t n, int64_t k,
                           cudaStream_t stream) {
  const int64_t total = (n / kTileN) * (k / kStageK) * (kTileN * kGroupsPerRow);
  auto* o = static_cast<uint16_t*>(out);
  if (fmt == kNVFP4)
    dequant_kernel<kNVFP4><<<grid_for(total), kThreads, 0, stream>>>(rep, o, n, k);
  else if (fmt == kNVFP4F16)
    dequant_kernel<kNVFP4F16><<<grid_for(total), kThreads, 0, stream>>>(rep, o, n, k);
  else
    dequant_kernel<kMXFP4><<<grid_for(total), kThreads, 0, stream>>>(rep, o, n, k);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace petit
