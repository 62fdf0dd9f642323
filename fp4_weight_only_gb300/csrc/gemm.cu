// BF16 x FP4 weight-only GEMM for sm_103a (tcgen05 + tensor memory).
//
//   C[m, n] = alpha * sum_k A[m, k] * W'[n, k]
//
// W' is the register-dequantised weight (Wq * 2^-8 for NVFP4, Wq for MXFP4)
// and alpha the matching epilogue factor (g * 2^8, or 1).
//
// Design (one CTA per SM, persistent, stream-K):
// * The MMA runs "swap-AB": 128 weight rows fill the tcgen05 M side, the m
//   activation rows are the N side (16..128), so decode-sized m does not waste
//   the tensor core (the pages' small-m, memory-bound regime: Petit blog,
//   "Performance results").
// * Work = (weight tile, activation tile, 128-k stage) units in tile-major
//   order, split evenly over the CTAs; a CTA's range covers at most two
//   partial tiles, whose FP32 partial sums go to the workspace.  The last CTA
//   to finish a shared tile (atomic arrival counter, no waiting) adds the
//   partials in a fixed order and writes C, so results are deterministic.
// * Warp roles:
//     warp 0      producer: bulk copies of the repacked FP4 chunk and its
//                 scales, and two 2-D TMA boxes of A (128-byte swizzle), into
//                 a ring of shared-memory stages (mbarrier full/empty);
//     warp 1      tensor-memory owner and MMA issuer (one thread);
//     warps 2-5   epilogue: tensor memory -> registers -> C or partials;
//     warps 6-13  dequantisers: shared memory -> registers -> BF16 -> tensor
//                 memory, where the MMA reads its A operand.  Each thread owns
//                 one weight row (= one tensor-memory lane).
//   Keeping the dequantised weights in tensor memory avoids writing 2 bytes
//   per weight back to shared memory, so shared-memory bandwidth only carries
//   the FP4 chunk and the activation tile.
// * Every wait is bounded; a wait that runs out records a timeout in the
//   workspace status word and the CTA shuts down cleanly.
#include <cuda_bf16.h>

#include "fp4_layout.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace petit {
namespace {

constexpr int kThreads = 448;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;    // warps 2..5
constexpr int kDeqWarp0 = 6;    // warps 6..13
constexpr int kNumDeqWarps = 8;
constexpr int kNumABufs = 4;    // dequantised-weight buffers in tensor memory
constexpr int kAColsPerBuf = kStageK / 2;  // 64 columns of BF16x2 per stage
constexpr int kDColBase = kNumABufs * kAColsPerBuf;  // 256
constexpr uint32_t kTmemCols = 512;

struct Params {
  const uint8_t* w;
  const uint8_t* s;
  __nv_bfloat16* c;
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  int32_t m, n;
  int32_t m_tiles, k_stages;
  int64_t units;
  int32_t num_ctas;
  float alpha;
  uint64_t timeout_ns;
};

template <int FMT, int BN>
struct Cfg {
  static constexpr int kAHalfBytes = BN * 128;           // 64 k x BN rows, swizzled
  static constexpr int kABytes = 2 * kAHalfBytes;
  static constexpr int kSBytes = FmtTraits<FMT>::kSChunkBytes;
  static constexpr int kStageBytes = kABytes + kWChunkBytes + kSBytes;
  static constexpr int kStages0 = (212 * 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 12 ? 12 : kStages0;
  static constexpr int kTx = kStageBytes;
  static constexpr int kNumD = 2;                        // accumulator buffers
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 512;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N");
  static_assert(kDColBase + kNumD * BN <= static_cast<int>(kTmemCols), "tensor memory");
  static_assert(kStages >= 2, "pipeline depth");
};

// CTA that owns stream-K unit u when U units are split over P CTAs with
// CTA c covering [floor(c U / P), floor((c+1) U / P)).
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t U, int64_t P) {
  return ((u + 1) * P + U - 1) / U - 1;
}

template <int FMT, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap_a) {
  using C = Cfg<FMT, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;
  uint8_t* sm_w = sm_a + C::kStages * C::kABytes;
  uint8_t* sm_s = sm_w + C::kStages * kWChunkBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm_s + C::kStages * C::kSBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* afull = empty + C::kStages;
  uint64_t* aempty = afull + kNumABufs;
  uint64_t* dfull = aempty + kNumABufs;
  uint64_t* dempty = dfull + C::kNumD;
  uint64_t* fin = dempty + C::kNumD;
  uint64_t* epi_bar = fin + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(epi_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* epi_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t U = p.units;
  const int64_t P = p.num_ctas;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = cta * U / P;
  const int64_t u1 = (cta + 1) * U / P;
  const int64_t KS = p.k_stages;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kNumDeqWarps + 1);
    }
    for (int i = 0; i < kNumABufs; ++i) {
      mbar_init(smem_u32(&afull[i]), kNumDeqWarps);
      mbar_init(smem_u32(&aempty[i]), 1);
    }
    for (int i = 0; i < C::kNumD; ++i) {
      mbar_init(smem_u32(&dfull[i]), 1);
      mbar_init(smem_u32(&dempty[i]), 4);
    }
    mbar_init(smem_u32(fin), 1);
    mbar_init(smem_u32(epi_bar), 4);
    *abort_flag = 0;
    *epi_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) tma_prefetch_desc(&tmap_a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  auto fail = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(smem_u32(bar), parity, p.timeout_ns, abort_flag)) return true;
    if (!*abort_flag) fail();
    return false;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int64_t issued = 0;
      for (int64_t u = u0; u < u1; ++u, ++issued) {
        const int st = static_cast<int>(issued % C::kStages);
        const uint32_t ph = static_cast<uint32_t>((issued / C::kStages) & 1);
        if (!wait(&empty[st], ph ^ 1u)) break;
        const int64_t tile = u / KS, ks = u % KS;
        const int64_t nt = tile / p.m_tiles, mt = tile % p.m_tiles;
        const uint32_t fb = smem_u32(&full[st]);
        mbar_arrive_expect_tx(fb, C::kTx);
        bulk_g2s(smem_u32(sm_w + st * kWChunkBytes), p.w + w_chunk_offset(nt, ks, KS),
                 kWChunkBytes, fb, policy);
        bulk_g2s(smem_u32(sm_s + st * C::kSBytes),
                 p.s + static_cast<size_t>(nt * KS + ks) * C::kSBytes, C::kSBytes, fb, policy);
        const uint32_t a_dst = smem_u32(sm_a + st * C::kABytes);
        tma_load_2d(a_dst, &tmap_a, static_cast<int32_t>(ks * kStageK),
                    static_cast<int32_t>(mt * BN), fb);
        tma_load_2d(a_dst + C::kAHalfBytes, &tmap_a, static_cast<int32_t>(ks * kStageK + 64),
                    static_cast<int32_t>(mt * BN), fb);
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        const int64_t first = issued > C::kStages ? issued - C::kStages : 0;
        for (int64_t j = first; j < issued; ++j)
          mbar_wait_bounded(smem_u32(&full[j % C::kStages]), (j / C::kStages) & 1, p.timeout_ns,
                            nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int64_t i = 0;
      int64_t seg = 0;
      for (int64_t u = u0; u < u1; ++u, ++i) {
        const int st = static_cast<int>(i % C::kStages);
        const uint32_t ph = static_cast<uint32_t>((i / C::kStages) & 1);
        const int b = static_cast<int>(i % kNumABufs);
        const uint32_t pb = static_cast<uint32_t>((i / kNumABufs) & 1);
        const bool first = (u == u0) || (u % KS == 0);
        const bool last = (u == u1 - 1) || (u % KS == KS - 1);
        const int d = static_cast<int>(seg % C::kNumD);
        if (first && !wait(&dempty[d], static_cast<uint32_t>(((seg / C::kNumD) & 1) ^ 1))) break;
        if (!wait(&full[st], ph)) break;
        if (!wait(&afull[b], pb)) break;
        tc_fence_after();
        const uint32_t a_smem = smem_u32(sm_a + st * C::kABytes);
        const uint32_t d_tmem = tmem + kDColBase + d * BN;
#pragma unroll
        for (int j = 0; j < kStageK / 16; ++j) {
          const uint64_t bdesc =
              smem_desc_kmajor_sw128(a_smem + (j >> 2) * C::kAHalfBytes) + (((j & 3) * 32) >> 4);
          mma_ts_f16(d_tmem, tmem + b * kAColsPerBuf + j * 8, bdesc, C::kIdesc,
                     (first && j == 0) ? 0u : 1u);
        }
        mma_commit(smem_u32(&empty[st]));
        mma_commit(smem_u32(&aempty[b]));
        if (last) {
          mma_commit(smem_u32(&dfull[d]));
          ++seg;
        }
      }
      // all issued MMAs complete before tensor memory is released
      mma_commit(smem_u32(fin));
      mbar_wait_bounded(smem_u32(fin), 0, p.timeout_ns, nullptr);
    }
  } else if (warp < kDeqWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const int epi_tid = threadIdx.x - kEpiWarp0 * 32;
    int64_t seg = 0;
    const int64_t first_tile_of_cta = u0 / KS;
    uint32_t epi_phase = 0;
    // bounded barrier among the four epilogue warps (a hardware named
    // barrier has no time limit)
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(epi_bar));
      const bool ok = wait(epi_bar, epi_phase & 1u);
      ++epi_phase;
      return ok;
    };
    for (int64_t u = u0; u < u1; ++seg) {
      const int64_t tile = u / KS;
      const int64_t seg_end = (tile + 1) * KS < u1 ? (tile + 1) * KS : u1;
      const bool full_tile = (u == tile * KS) && (seg_end == (tile + 1) * KS);
      const int64_t nt = tile / p.m_tiles, mt = tile % p.m_tiles;
      const int d = static_cast<int>(seg % C::kNumD);
      if (!wait(&dfull[d], static_cast<uint32_t>((seg / C::kNumD) & 1))) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + kDColBase + d * BN;
      const int64_t ncol = static_cast<int64_t>(nt) * kTileN + r;
      const int64_t slot = 2 * cta + (tile == first_tile_of_cta ? 0 : 1);
      float* my_slot = p.partials + static_cast<size_t>(slot) * (BN * kTileN);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(tbase + c0, v);
        tmem_wait_ld();
        if (full_tile) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t mrow = static_cast<int64_t>(mt) * BN + c0 + j;
            if (mrow < p.m)
              p.c[mrow * p.n + ncol] = __float2bfloat16_rn(p.alpha * __uint_as_float(v[j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) my_slot[(c0 + j) * kTileN + r] = __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&dempty[d]));
      if (!full_tile) {
        // stream-K fix-up: the last contributor sums all partials in CTA order
        const int64_t c_first = cta_of_unit(tile * KS, U, P);
        const int64_t c_last = cta_of_unit((tile + 1) * KS - 1, U, P);
        __threadfence();
        if (!epi_sync()) break;
        if (epi_tid == 0) {
          const uint32_t old = atomicAdd(&p.counters[tile], 1u);
          const int is_last = (static_cast<int64_t>(old) == c_last - c_first);
          if (is_last) atomicExch(&p.counters[tile], 0u);  // ready for the next call
          *epi_flag = is_last;
        }
        if (!epi_sync()) break;
        if (*epi_flag) {
          __threadfence();
#pragma unroll 1
          for (int col = 0; col < BN; ++col) {
            const int64_t mrow = static_cast<int64_t>(mt) * BN + col;
            if (mrow >= p.m) break;
            float acc = 0.0f;
            for (int64_t c = c_first; c <= c_last; ++c) {
              const int64_t cs = 2 * c + ((c * U / P) / KS == tile ? 0 : 1);
              acc += ld_cg_f32(p.partials + static_cast<size_t>(cs) * (BN * kTileN) +
                               col * kTileN + r);
            }
            p.c[mrow * p.n + ncol] = __float2bfloat16_rn(p.alpha * acc);
          }
        }
        if (!epi_sync()) break;
      }
      u = seg_end;
    }
  } else {
    // ---------------------------------------------------------- dequantise
    const int dw = warp - kDeqWarp0;
    const int h = dw >> 2;          // which 64-k half of the stage
    const int q = warp & 3;         // tensor-memory lane quarter
    const int r = 32 * q + lane;    // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    int64_t i = 0;
    for (int64_t u = u0; u < u1; ++u, ++i) {
      const int st = static_cast<int>(i % C::kStages);
      const uint32_t ph = static_cast<uint32_t>((i / C::kStages) & 1);
      const int b = static_cast<int>(i % kNumABufs);
      const uint32_t pb = static_cast<uint32_t>((i / kNumABufs) & 1);
      if (!wait(&full[st], ph)) break;
      if (!wait(&aempty[b], pb ^ 1u)) break;
      const uint8_t* wsm = sm_w + st * kWChunkBytes;
      const uint4 g0 = *reinterpret_cast<const uint4*>(wsm + ((2 * h) * kTileN + r) * 16);
      const uint4 g1 = *reinterpret_cast<const uint4*>(wsm + ((2 * h + 1) * kTileN + r) * 16);
      uint32_t sc0, sc1;
      if constexpr (FMT == kNVFP4) {
        const uint32_t v =
            *reinterpret_cast<const uint32_t*>(sm_s + st * C::kSBytes + (h * kTileN + r) * 4);
        sc0 = v & 0xFFFFu;
        sc1 = v >> 16;
      } else {
        const uint32_t v =
            *reinterpret_cast<const uint16_t*>(sm_s + st * C::kSBytes + (h * kTileN + r) * 2);
        sc0 = v & 0xFFu;
        sc1 = v >> 8;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
      uint32_t o0[16], o1[16];
      decode_group<FMT>(g0, sc0, o0);
      decode_group<FMT>(g1, sc1, o1);
      const uint32_t acol = tmem + lane_base + b * kAColsPerBuf + (2 * h) * 16;
      tmem_st_x16(acol, o0);
      tmem_st_x16(acol + 16, o1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&afull[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int FMT, int BN>
cudaError_t launch_t(const Params& prm, const CUtensorMap& tmap, cudaStream_t stream) {
  using C = Cfg<FMT, BN>;
  static int attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(gemm_kernel<FMT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(prm.num_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<FMT, BN>, prm, tmap);
}

template <int FMT>
cudaError_t launch_fmt(int bn, const Params& prm, const CUtensorMap& tmap, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_t<FMT, 16>(prm, tmap, s);
    case 32: return launch_t<FMT, 32>(prm, tmap, s);
    case 64: return launch_t<FMT, 64>(prm, tmap, s);
    case 128: return launch_t<FMT, 128>(prm, tmap, s);
    default: return cudaErrorInvalidValue;
  }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

GemmPlan plan_gemm(int64_t m, int64_t n, int64_t k, int fmt, int num_sms) {
  GemmPlan pl{};
  pl.fmt = fmt;
  pl.bn = m <= 16 ? 16 : (m <= 32 ? 32 : (m <= 64 ? 64 : 128));
  pl.m_tiles = static_cast<int>((m + pl.bn - 1) / pl.bn);
  pl.n_tiles = static_cast<int>(n / kTileN);
  pl.k_stages = static_cast<int>(k / kStageK);
  pl.units = static_cast<int64_t>(pl.n_tiles) * pl.m_tiles * pl.k_stages;
  pl.num_ctas = static_cast<int>(pl.units < num_sms ? pl.units : num_sms);
  if (pl.num_ctas < 1) pl.num_ctas = 1;
  pl.ws.counters_off = kWsHeaderBytes;
  pl.ws.partials_off =
      align_up(pl.ws.counters_off + sizeof(uint32_t) * static_cast<size_t>(pl.n_tiles) * pl.m_tiles, 256);
  pl.ws.total = pl.ws.partials_off +
                sizeof(float) * 2ull * static_cast<size_t>(pl.num_ctas) * pl.bn * kTileN;
  return pl;
}

cudaError_t launch_gemm(const GemmPlan& pl, const GemmArgs& a, const CUtensorMap& tmap,
                        cudaStream_t stream) {
  Params prm{};
  prm.w = a.w;
  prm.s = a.s;
  prm.c = static_cast<__nv_bfloat16*>(a.C);
  prm.partials = reinterpret_cast<float*>(a.workspace + pl.ws.partials_off);
  prm.counters = reinterpret_cast<uint32_t*>(a.workspace + pl.ws.counters_off);
  prm.status = reinterpret_cast<uint32_t*>(a.workspace);
  prm.m = static_cast<int32_t>(a.m);
  prm.n = static_cast<int32_t>(a.n);
  prm.m_tiles = pl.m_tiles;
  prm.k_stages = pl.k_stages;
  prm.units = pl.units;
  prm.num_ctas = pl.num_ctas;
  prm.alpha = a.alpha;
  prm.timeout_ns = a.timeout_ns;
  if (pl.fmt == kNVFP4) return launch_fmt<kNVFP4>(pl.bn, prm, tmap, stream);
  return launch_fmt<kMXFP4>(pl.bn, prm, tmap, stream);
}

}  // namespace petit
