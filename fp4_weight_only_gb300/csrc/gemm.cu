// BF16 x FP4 weight-only GEMM for sm_103a (tcgen05 + tensor memory).
//
//   C[m, n] = alpha * sum_k A[m, k] * W'[n, k]
//
// W' is the register-dequantised weight (Wq * 2^-8 for NVFP4, Wq for MXFP4)
// and alpha the matching epilogue factor (g * 2^8, or 1).
//
// Design (one CTA per SM, persistent, stream-K):
// * The MMA runs "swap-AB": 128 weight rows fill the tcgen05 M side, the m
//   activation rows are the N side (16..256), so decode-sized m does not waste
//   the tensor core (the pages' small-m, memory-bound regime: Petit blog,
//   "Performance results").
// * Work = (weight tile, activation tile, 128-k stage) units in tile-major
//   order, split over the CTAs in contiguous ranges (stream-K); a CTA's range
//   covers at most two partial tiles, whose FP32 partial sums go to the
//   workspace.  The last CTA to finish a shared tile (atomic arrival counter,
//   no waiting) adds the partials in a fixed order and writes C, so results
//   are deterministic.
// * CTA pairs (PAIR, for 128/256-row activation tiles): two CTAs of a
//   cluster take adjacent 128-row weight tiles of one 256-row work tile and
//   one thread of the even CTA issues cta_group::2 MMAs (M = 256); each CTA
//   holds half of the activation rows.  The odd CTA's warp 1 forwards its
//   activation-stage completions; its dequantisers and epilogue arrive on the
//   even CTA's barriers; MMA completions are committed to both CTAs.
// * A pipeline unit is KU (1 or 2) consecutive 128-k chunks of one tile.
//   Its data arrives with exactly two copies: one bulk copy of the repacked
//   codes + scales (contiguous) and one 3-D TMA box holding all 2*KU 64-k
//   slabs of A.  The TMA unit of an SM sustains only a limited number of
//   requests per microsecond, so few large requests keep HBM busy.
// * Warp roles:
//     warp 0      producer: the two copies per unit into a ring of
//                 shared-memory stages (mbarrier full/empty);
//     warps 1, 14, 15  tensor-memory owner (warp 1) and MMA issuers (one
//                 elected lane each; one issuer at N = 64, 256 and in pairs);
//     warps 2-5   epilogue: tensor memory -> registers -> C or partials
//                 (128/256-row tiles: C through a 16-row shared-memory stage,
//                 in whole 256-byte row segments);
//     warps 6-13  dequantisers: shared memory -> registers -> BF16 -> tensor
//                 memory, where the MMA reads its A operand.  Each thread owns
//                 one weight row (= one tensor-memory lane).
//   Keeping the dequantised weights in tensor memory avoids writing 2 bytes
//   per weight back to shared memory, so shared-memory bandwidth only carries
//   the FP4 chunk and the activation tile.
// * Every wait is bounded; a wait that runs out records a timeout in the
//   workspace status word and the CTA shuts down cleanly.
// * Bounds-checking build (-DPETIT_CHECK_BOUNDS, a separate library): every
//   global-memory access, bulk or tensor copy and shared- or tensor-memory
//   buffer index of the kernel is checked against its buffer's extent first.
//   A failed check skips the access (a skipped copy still arrives on its
//   barrier, so no wait is left hanging on it), marks the CTA aborted and
//   the CTA shuts down as after a timeout; thread 0 then records
//   kStatusBounds in the workspace status word.  No trap, no assert.  In the
//   normal build each check is the constant true and its operand is not
//   compiled.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fp4_layout.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace petit {
namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;     // tensor-memory owner and MMA issuer 0
constexpr int kEpiWarp0 = 2;    // warps 2..5
constexpr int kDeqWarp0 = 6;    // dequantiser warps 6 .. 6 + 4 * groups - 1
constexpr int kDeqGroupWarps = 4;   // one dequantiser group: a warp per lane quarter
constexpr int kMaxMmaThreads = 3;
constexpr uint32_t kTmemCols = 512;
constexpr int kFixBatch = 2;   // split-tile contributors whose partials are loaded together
// bits of a CTA's abort flag (shared memory)
constexpr int kAbortTimeout = 1;
constexpr int kAbortBounds = 2;

#ifdef PETIT_CHECK_BOUNDS
// A failed index check aborts the CTA.
__device__ __forceinline__ bool check_ok(bool ok, volatile int* abort) {
  if (!ok) atomicOr(const_cast<int*>(abort), kAbortBounds);
  return ok;
}
#define PETIT_CHECK(cond) check_ok((cond), abort_flag)
#else
#define PETIT_CHECK(cond) true
#endif

struct Params {
  const uint8_t* rep;
  uint16_t* c;              // BF16 (or FP16 for the FP16 layout) [rows][n]
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  int32_t n, n_tiles;
  int32_t k_units;          // units per tile = k / (128 * KU)
  int64_t units;
  int32_t num_ctas;
  int32_t units_q, units_r; // units / num_ctas, units % num_ctas
  int32_t use_bounds;       // CTA c covers [bound[c], bound[c+1]) (else an even split)
  int32_t bound[kMaxBoundCtas + 1];
  int32_t weights_reused;   // a group has several activation tiles
  uint64_t timeout_ns;
  const float* alpha_dev;   // nullable: device-resident factor, times alpha_scale
  float alpha_scale;
  int64_t rep_stride;       // bytes between groups' repacked weights
  int32_t num_groups;
  int32_t row_off[kMaxGroups + 1];    // group g: activation / output rows
  int32_t tile_base[kMaxGroups + 1];  // group g: first tile
  float group_alpha[kMaxGroups];      // epilogue factor per group
#ifdef PETIT_CHECK_BOUNDS
  int64_t chk_rep_bytes;   // bytes of each group's repacked weights the kernel may read
  int64_t chk_c_elems;     // elements of C it may write
  int32_t chk_a_rows;      // activation rows (the tensor map's row extent)
#endif
};

// Split tiles.  A contributor stores its FP32 partial and then arrives on
// the tile's counter (acq_rel); the last to arrive adds all partials in CTA
// order and writes C, so the result is the same whichever CTA sums, and no
// CTA ever waits for another.  A CTA's last segment is usually the
// beginning of a tile whose other contributors ran their parts at the start
// of their ranges: if the counter (an acquire load, before and again after
// the segment's MMAs) already shows every other contributor, this CTA is
// the last one without arriving, so it stores nothing and adds its
// accumulator straight from tensor memory.
//
// When the summed tile is the CTA's last segment the sum is deferred to
// after the kernel's final barrier, so that every warp shares it: with
// BN = 256 the tile's partials are 128 KB per contributor.
struct FixJob {
  uint16_t* c_g;                        // output rows of the tile's group
  int64_t c_first, c_last, first_slot;  // contributing CTAs, slot of the first
  int64_t row0, col0, g_rows;           // tile origin in C; rows of the group
  float alpha;
  int32_t d;                            // accumulator buffer of the segment
  uint32_t has;                         // bit t: issuer t's accumulator contributes
  int32_t valid;
};

// Position of a tile: group, weight tile, activation tile (tile-major in a
// group, groups in order).  Walked tile by tile without divisions.
struct TileCursor {
  int32_t g;
  int32_t m_tiles;   // activation tiles of group g
  int32_t nt, mt;
  int32_t row0;      // first activation row of group g
};

template <int BN>
__device__ __forceinline__ int32_t group_m_tiles(const Params& p, int g) {
  return (p.row_off[g + 1] - p.row_off[g] + BN - 1) / BN;
}

template <int BN>
__device__ __forceinline__ TileCursor cursor_at(const Params& p, int64_t tile) {
  TileCursor c;
  c.g = 0;
  while (c.g + 1 < p.num_groups && p.tile_base[c.g + 1] <= tile) ++c.g;
  c.m_tiles = group_m_tiles<BN>(p, c.g);
  c.row0 = p.row_off[c.g];
  const int32_t local = static_cast<int32_t>(tile - p.tile_base[c.g]);
  c.nt = c.m_tiles > 0 ? local / c.m_tiles : 0;
  c.mt = c.m_tiles > 0 ? local - c.nt * c.m_tiles : 0;
  return c;
}

template <int BN>
__device__ __forceinline__ void cursor_next(const Params& p, TileCursor& c) {
  if (++c.mt < c.m_tiles) return;
  c.mt = 0;
  if (++c.nt < p.n_tiles) return;
  c.nt = 0;
  do {
    ++c.g;
  } while (c.g < p.num_groups && group_m_tiles<BN>(p, c.g) == 0);
  c.m_tiles = c.g < p.num_groups ? group_m_tiles<BN>(p, c.g) : 0;
  c.row0 = c.g < p.num_groups ? p.row_off[c.g] : 0;
}

// The weight-chunk stream of a CTA: unit by unit, the unit's KU repacked
// chunks (contiguous codes + scales) by one bulk copy into the next weight
// stage.  Addresses advance incrementally (a runtime 64-bit division costs
// hundreds of cycles in a single thread): the consecutive units of a tile
// are adjacent chunks, so the source moves on by one unit's bytes and is
// recomputed only at a tile boundary; stage addresses move on by one stage
// and wrap.
template <int FMT, int BN, int KU>
struct WeightStream {
  static constexpr uint32_t kBytes = KU * FmtTraits<FMT>::kChunkBytes;
  const uint8_t* src;
  int32_t KS;            // units per tile
  int32_t ku;            // unit index inside the tile
  int32_t wmul, wadd;    // weight tile of work tile nt: nt * wmul + wadd (CTA pairs: 2 nt + rank)
  TileCursor cur;
  uint32_t dst, dst0;    // shared-memory stage, first stage
  uint32_t bar, full0;   // stage * 8, address of the stage-0 full barrier
  uint32_t ph;           // phase of the stage's free barrier to wait for, ^ 1
  int32_t stages;

  // starting at unit ku of tile `tile`
  __device__ __forceinline__ void init(const Params& p, int32_t tile, int32_t ku0, int32_t ks,
                                       uint32_t sm_w, uint32_t wfull0, int32_t nstages,
                                       int32_t tile_mul = 1, int32_t tile_add = 0) {
    KS = ks;
    ku = ku0;
    wmul = tile_mul;
    wadd = tile_add;
    cur = cursor_at<BN>(p, tile);
    src = p.rep + cur.g * p.rep_stride +
          chunk_offset<FMT>(cur.nt * wmul + wadd, ku * KU, KS * KU);
    dst = dst0 = sm_w;
    bar = 0;
    full0 = wfull0;
    ph = 0;
    stages = nstages;
  }
  __device__ __forceinline__ void advance(const Params& p) {
    src += kBytes;
    dst += kBytes;
    bar += 8;
    if (bar == 8u * stages) {
      bar = 0;
      dst = dst0;
      ph ^= 1u;
    }
    if (++ku == KS) {
      ku = 0;
      cursor_next<BN>(p, cur);
      src = p.rep + cur.g * p.rep_stride + chunk_offset<FMT>(cur.nt * wmul + wadd, 0, KS * KU);
    }
  }
  __device__ __forceinline__ void issue(const Params& p, uint64_t policy) {
    mbar_arrive_expect_tx(full0 + bar, kBytes);
    bulk_g2s(dst, src, kBytes, full0 + bar, policy);
    advance(p);
  }
  // bounds-checking build: the copy's source lies inside its group's
  // repacked weights and its destination inside the weight ring
  __device__ __forceinline__ bool in_bounds(const Params& p) const {
#ifdef PETIT_CHECK_BOUNDS
    if (cur.g < 0 || cur.g >= p.num_groups) return false;
    const uint8_t* base = p.rep + cur.g * p.rep_stride;
    return src >= base && src + kBytes <= base + p.chk_rep_bytes && dst >= dst0 &&
           dst + kBytes <= dst0 + static_cast<uint32_t>(stages) * kBytes &&
           bar < 8u * static_cast<uint32_t>(stages);
#else
    return true;
#endif
  }
  // a copy that failed its check: the stage's barrier completes without data
  __device__ __forceinline__ void skip(const Params& p) {
    mbar_arrive(full0 + bar);
    advance(p);
  }
};

template <int FMT, int BN, int KU, bool PAIR = false>
struct Cfg {
  using T = FmtTraits<FMT>;
  // CTA pairs (PAIR): two CTAs of a cluster take adjacent 128-row weight
  // tiles of the same work tile and one thread of the even CTA issues
  // cta_group::2 MMAs (M = 256); each CTA holds BN / 2 of the tile's BN
  // activation rows, so a CTA's activation stage and its share of the L2
  // activation traffic are halved.
  static constexpr int kARows = PAIR ? BN / 2 : BN;            // activation rows in this CTA
  static constexpr int kAHalfBytes = kARows * 128;             // one 64-k slab
  static constexpr int kABytes = 2 * KU * kAHalfBytes;
  static constexpr int kWBytes = KU * T::kChunkBytes;          // codes + scales
  // MMA-issuing threads.  A thread issues one tcgen05.mma per ~65 cycles
  // whatever N is, so short (N <= 32) MMAs need several issuers on
  // different SM sub-partitions.  They take the CTA's units round-robin,
  // each into its own accumulator, which the epilogue adds in a fixed order.
  // Three issuers (warps 1, 14, 15 on sub-partitions 1, 2, 3) keep the CTA
  // at 16 warps, four per sub-partition, so each thread may use 128 registers.
  // At N = 64 one issuer leaves room for two accumulators, so a tile's
  // epilogue overlaps the next tile's MMAs (measured on GB300: gate_up at
  // m = 64 12 % faster than with two issuers and one accumulator each); at
  // N = 128 two issuers stay faster.
  static constexpr int kMmaThreads = PAIR ? 1 : BN <= 32 ? 3 : BN == 128 ? 2 : 1;
  // dequantiser groups (four warps each) taking units round-robin
  static constexpr int kDeqGroups = 2;
  static constexpr int kMmaWarpX = kDeqWarp0 + kDeqGroupWarps * kDeqGroups - 1;  // issuer t>=1: +t
  static constexpr int kThreads = 32 * (kMmaWarpX + kMmaThreads);
  static constexpr int kAColsPerUnit = KU * (kStageK / 2);     // BF16x2 columns
  // accumulator buffers per issuer: two when they fit beside three A-buffers
  // (the epilogue of one tile then overlaps the next tile's MMAs)
  static constexpr int kNumD =
      kMmaThreads * 2 * BN + 3 * kAColsPerUnit <= static_cast<int>(kTmemCols) ? 2 : 1;
  static constexpr int kNumA0 =
      (static_cast<int>(kTmemCols) - kMmaThreads * kNumD * BN) / kAColsPerUnit;
  // Every mbarrier is waited on by one fixed consumer that waits for each of
  // its phases in turn: a parity wait cannot tell phase j from phase j + 2,
  // so a consumer that skipped a phase could pass a wait on a phase that has
  // not completed.  The two dequantiser groups take units by parity, the
  // MMA issuers by unit index modulo kMmaThreads; hence
  //   * kWStages is even (a weight stage always holds units of one parity);
  //   * kXStages is a multiple of kMmaThreads (an activation stage always
  //     feeds the same issuer) and, with several issuers, even: the
  //     dequantisers also wait on the activation stage's mdone barrier to
  //     reuse an A-buffer, so its units must belong to one group;
  //   * kNumA is a multiple of kMmaThreads (an A-buffer always feeds the
  //     same issuer) and at most kXStages: the dequantiser waits for mdone of
  //     unit i - kNumA, and no later unit sharing that barrier may complete
  //     first.
  static constexpr int kXMult = kMmaThreads == 3 ? 6 : kMmaThreads;
  static constexpr int kXBudget =
      PAIR ? (BN >= 256 ? 128 * 1024 : 96 * 1024)
           : (BN >= 256 ? 192 * 1024 : (BN <= 32 ? 96 * 1024 : 128 * 1024));
  static constexpr int kXStages0 = (kXBudget / kABytes) / kXMult * kXMult;
  static constexpr int kXStages = kXStages0 > 16 ? 16 / kXMult * kXMult : kXStages0;
  static constexpr int kRingBytes = 220 * 1024;
  static constexpr int kWStages0 =
      (kRingBytes - kXStages * kABytes) / kWBytes / kDeqGroups * kDeqGroups;
  static constexpr int kWStages = kWStages0 > 12 ? 12 : kWStages0;
  static constexpr int kNumA1 = (kNumA0 > 4 ? 4 : kNumA0) / kMmaThreads * kMmaThreads;
  static constexpr int kNumA = kNumA1 > kXStages ? kXStages / kMmaThreads * kMmaThreads : kNumA1;
  static constexpr int kDColBase = kNumA * kAColsPerUnit;      // D(t, d) at + (t*kNumD+d)*BN
  // 128/256-row tiles: 16 output rows x 128 columns of BF16 staged in
  // shared memory, so that C is written in whole 256-byte row segments
  static constexpr int kStageC = BN >= 128 ? 16 * kTileN * 2 : 0;
  static constexpr int kSmemBytes =
      1024 + kXStages * kABytes + kWStages * kWBytes + 1024 + kStageC;
  static constexpr uint32_t kM = PAIR ? 256 : 128;   // MMA M (weight rows of both CTAs)
  static constexpr uint32_t kIdesc =
      FMT == kNVFP4F16 ? idesc_f16_f32(kM, BN) : idesc_bf16_f32(kM, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(!PAIR || (BN >= 128 && KU == 1), "CTA pairs: 128- or 256-row tiles, 128-k units");
  static_assert(kNumA >= 2, "tensor memory");
  static_assert(kDColBase + kMmaThreads * kNumD * BN <= static_cast<int>(kTmemCols),
                "tensor memory");
  static_assert(kMmaThreads <= kMaxMmaThreads, "issuers");
  static_assert(kWStages >= 2 && kXStages >= 2 && kWStages % kDeqGroups == 0, "pipeline depth");
  static_assert(kXStages % kMmaThreads == 0 && (kMmaThreads == 1 || kXStages % kDeqGroups == 0) &&
                    kNumA % kMmaThreads == 0 && kNumA <= kXStages,
                "fixed consumer per barrier");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // tcgen05.alloc of all 512 tensor-memory columns blocks (in hardware, with
  // no time limit) until the columns are free.  It never waits here because
  // no two CTAs of this kernel fit on one SM: each takes more than half of
  // the SM's 228 KB of shared memory, so the next launch's CTA (under
  // programmatic dependent launch) starts on an SM only after this one has
  // exited and freed its columns.
  static_assert(2 * kSmemBytes > 228 * 1024, "one CTA per SM");
  // barriers, tensor-memory holder, flags and the deferred fix-up job fit in
  // the 1024 bytes after the rings
  static_assert((2 * kWStages + 3 * kXStages + kNumA + 2 * kNumD + kMaxMmaThreads + 1) * 8 + 16 +
                        sizeof(FixJob) + 16 <= 1024,
                "barrier region");
};

// Output element bits: BF16, or FP16 for the FP16-activation layout (RNE).
template <int FMT>
__device__ __forceinline__ uint16_t out_bits(float x) {
  if constexpr (FMT == kNVFP4F16) return __half_as_ushort(__float2half_rn(x));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// First unit of CTA c's stream-K range (c = P: the end of the last).  An
// even split is floor(c U / P) = c q + c r / P with q = U / P, r = U % P;
// c r < P^2 fits 32 bits, so no 64-bit division is needed (this sits before
// the producer's first activation copy, on the critical path of the CTAs
// that start last).
__device__ __forceinline__ int32_t cta_lo(const Params& p, int32_t c) {
  return p.use_bounds ? p.bound[c] : c * p.units_q + (c * p.units_r) / p.num_ctas;
}

// CTA whose stream-K range holds unit u.
__device__ __forceinline__ int32_t cta_of_unit(const Params& p, int64_t u) {
  if (!p.use_bounds)
    return static_cast<int32_t>(((u + 1) * p.num_ctas + p.units - 1) / p.units - 1);
  int lo = 0, hi = p.num_ctas - 1;   // the last c with bound[c] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.bound[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int FMT, int BN, int KU, bool PAIR>
__global__ void __launch_bounds__((Cfg<FMT, BN, KU, PAIR>::kThreads), 1)
    gemm_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap_a) {
  using C = Cfg<FMT, BN, KU, PAIR>;
  using T = FmtTraits<FMT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sm_a = smem;                                   // [stage][2*KU slabs][kARows][128 B]
  uint8_t* sm_w = sm_a + C::kXStages * C::kABytes;         // [stage][KU chunks]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm_w + C::kWStages * C::kWBytes);
  // Weights and activations of a unit share a stage index but have their
  // own barriers, so each part is released as soon as its reader is done:
  //   wfull[s] / wfree[s]: weight chunk landed / decoded by all dequantisers;
  //   xfull[s] / mdone[s]: activation tile landed / the unit's MMAs completed
  //   (mdone also frees the unit's tensor-memory A-buffer).
  // The weights, the long HBM stream, so turn over a stage per unit without
  // waiting for the tensor core.
  uint64_t* wfull = bars;
  uint64_t* wfree = wfull + C::kWStages;
  uint64_t* xfull = wfree + C::kWStages;
  uint64_t* mdone = xfull + C::kXStages;
  uint64_t* afull = mdone + C::kXStages;
  uint64_t* dfull = afull + C::kNumA;
  uint64_t* dempty = dfull + C::kNumD;
  uint64_t* fin = dempty + C::kNumD;   // one per MMA issuer
  uint64_t* epi_bar = fin + kMaxMmaThreads;
  // CTA pairs: xpeer[s] (even CTA) -- the odd CTA's half of activation stage
  // s has landed (forwarded by the odd CTA's warp 1)
  uint64_t* xpeer = epi_bar + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(xpeer + (PAIR ? C::kXStages : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* epi_flag = abort_flag + 1;
  FixJob* fix = reinterpret_cast<FixJob*>(
      (reinterpret_cast<uintptr_t>(epi_flag + 1) + 15) & ~static_cast<uintptr_t>(15));
  // output staging (kStageC bytes) after the 1024-byte barrier region
  uint16_t* stage_c = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(bars) + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  [[maybe_unused]] const int64_t P = p.num_ctas;   // work ranges (index checks)
  [[maybe_unused]] const int64_t NS = PAIR ? 2 * P : P;   // CTAs: counters, 2 partial slots each
  // CTA pairs: both CTAs of a cluster share work range cta = blockIdx / 2;
  // rank 1 takes the odd weight tile and the second half of the activation
  // rows of every work tile.  Counters and partial slots are per CTA:
  // sid(c) is this rank's CTA of work range c.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int64_t cta = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
  auto sid = [&](int64_t c) -> int64_t { return PAIR ? 2 * c + rank : c; };
  const int32_t wmul = PAIR ? 2 : 1;   // weight tile of work tile nt: nt * wmul + rank
  const int64_t u0 = cta_lo(p, static_cast<int32_t>(cta));
  const int64_t u1 = cta_lo(p, static_cast<int32_t>(cta) + 1);
  const int64_t KS = p.k_units;
  const int32_t ks32 = p.k_units;
  const int32_t tile0_32 = static_cast<int32_t>(u0) / ks32;         // u0 < 2^31
  const int32_t ku0_32 = static_cast<int32_t>(u0) - tile0_32 * ks32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kWStages; ++i) {
      mbar_init(smem_u32(&wfull[i]), 1);
      mbar_init(smem_u32(&wfree[i]), kDeqGroupWarps);
    }
    for (int i = 0; i < C::kXStages; ++i) {
      mbar_init(smem_u32(&xfull[i]), 1);
      mbar_init(smem_u32(&mdone[i]), 1);
    }
    // (CTA pairs: the even CTA's afull and dempty also count the odd CTA's
    // dequantiser and epilogue warps)
    for (int i = 0; i < C::kNumA; ++i)
      mbar_init(smem_u32(&afull[i]), kDeqGroupWarps * (PAIR ? 2 : 1));
    for (int i = 0; i < C::kNumD; ++i) {
      mbar_init(smem_u32(&dfull[i]), C::kMmaThreads);
      mbar_init(smem_u32(&dempty[i]), 4 * (PAIR ? 2 : 1));
    }
    for (int i = 0; i < kMaxMmaThreads; ++i) mbar_init(smem_u32(&fin[i]), 1);
    mbar_init(smem_u32(epi_bar), 4);
    if constexpr (PAIR)
      for (int i = 0; i < C::kXStages; ++i) mbar_init(smem_u32(&xpeer[i]), 1);
    *abort_flag = 0;
    *epi_flag = 0;
    fix->valid = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == kProducerWarp && lane == 0) tma_prefetch_desc(&tmap_a);
  tc_fence_before();
  // CTA pairs: neither CTA arrives on the other's barriers before both have
  // initialised them
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // Programmatic dependent launch.  The next kernel on the stream may begin
  // launching now; its CTAs take an SM only when this kernel's CTA on it has
  // exited (shared memory), so they never crowd out this grid.  Before the
  // grid dependency wait this kernel touches only its weights, which must not
  // be written by the kernel just before it on the stream (a documented
  // precondition): the first ring of weight chunks is copied and the first
  // units are dequantised into tensor memory while the previous kernel
  // finishes.  The threads that read activations or the device-resident
  // global scale, or write global memory, wait first.
  grid_launch_dependents();

  // a wait that runs out records the abort in shared memory only; thread 0
  // (which has passed the grid dependency wait) reports it at the end
  auto fail = [&]() { atomicOr(const_cast<int*>(abort_flag), kAbortTimeout); };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(smem_u32(bar), parity, p.timeout_ns, abort_flag)) return true;
    if (!*abort_flag) fail();
    return false;
  };
  // Waits in code that all 32 lanes of a warp run together, with warp
  // barriers and warp-collective tensor-memory stores after them, must give
  // every lane the same answer.  try_wait may suspend each lane on its own,
  // so a lane that checked the CTA's abort flag just as the phase completed
  // could leave the loop while the others go on, and they would then wait at
  // the next warp barrier without a time limit.  The dequantisers and the
  // epilogue therefore wait on the phase and the 2 s limit only (after an
  // abort elsewhere their phases stop completing, and every lane runs out
  // together); the MMA issuers and the activation forwarder, whose waits
  // cost little, vote instead and stop at once.
  auto wait_lane = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_wait_bounded(smem_u32(bar), parity, p.timeout_ns, nullptr)) return true;
    if (!*abort_flag) fail();
    return false;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait(bar, parity));
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // weights are streamed once (evict first) unless several m-tiles
      // revisit them, in which case the revisits should hit L2
      const uint64_t policy = p.weights_reused ? l2_policy_evict_normal() : l2_policy_evict_first();
      // Two streams over the same units: weight chunks (stage freed by the
      // dequantisers) and activation tiles (freed by the MMAs).  Whichever
      // has a free stage is issued next, weights first.  All per-unit
      // indices advance incrementally: a runtime 64-bit division costs
      // hundreds of cycles in a single thread.
      const int32_t nu = static_cast<int32_t>(u1 - u0);   // fewer than 2^31 units
      const int32_t ks = ks32;
      const int32_t tile0 = tile0_32;
      const int32_t ku0 = ku0_32;
      // the first ring of weight chunks was issued by an epilogue thread
      // before the grid dependency wait; this stream continues after it
      WeightStream<FMT, BN, KU> ws;
      ws.init(p, tile0, ku0, ks, smem_u32(sm_w), smem_u32(&wfull[0]), C::kWStages, wmul,
              static_cast<int32_t>(rank));
      int32_t wi = nu < C::kWStages ? nu : C::kWStages;
      for (int32_t j = 0; j < wi; ++j) ws.advance(p);
      int32_t xi = 0;
      uint32_t xph = 0;
      int32_t x_ku = ku0;
      TileCursor xc = cursor_at<BN>(p, tile0);
      // first activation row of this CTA's part of the tile (CTA pairs: the
      // odd CTA holds the second half)
      const int32_t xhalf = PAIR ? static_cast<int32_t>(rank) * C::kARows : 0;
      int32_t xrow = xc.row0 + xc.mt * BN + xhalf, xk = x_ku * 2 * KU;
      const uint32_t xdst0 = smem_u32(sm_a);
      const uint32_t wfree0 = smem_u32(&wfree[0]);
      const uint32_t mdone0 = smem_u32(&mdone[0]), xfull0 = smem_u32(&xfull[0]);
      uint32_t xdst = xdst0, xbar = 0;   // bar: stage * 8
      // activations may be written by the previous kernel on the stream
      grid_dependency_wait();
      const uint64_t t0 = global_timer_ns();
      for (uint32_t spin = 0; wi < nu || xi < nu;) {
        bool progress = false;
        if (wi < nu && mbar_test_wait(wfree0 + ws.bar, ws.ph ^ 1u)) {
          if (!PETIT_CHECK(ws.in_bounds(p))) {
            ws.skip(p);
            ++wi;
            break;
          }
          ws.issue(p, policy);
          ++wi;
          progress = true;
        }
        if (xi < nu && mbar_test_wait(mdone0 + xbar, xph ^ 1u)) {
          // the box's first row and slab lie inside A (rows past its end
          // read as zeros) and its destination inside the activation ring
          if (!PETIT_CHECK(xrow >= 0 && xrow - xhalf < p.chk_a_rows && xk >= 0 &&
                           xk + 2 * KU <= 2 * KU * ks && xdst >= xdst0 &&
                           xdst + C::kABytes <= xdst0 + C::kXStages * C::kABytes &&
                           xbar < 8u * C::kXStages)) {
            mbar_arrive(xfull0 + xbar);
            ++xi;
            break;
          }
          mbar_arrive_expect_tx(xfull0 + xbar, C::kABytes);
          tma_load_3d(xdst, &tmap_a, 0, xrow, xk, xfull0 + xbar);
          ++xi;
          xk += 2 * KU;
          xdst += C::kABytes;
          xbar += 8;
          if (xbar == 8 * C::kXStages) {
            xbar = 0;
            xdst = xdst0;
            xph ^= 1u;
          }
          if (++x_ku == ks) {
            x_ku = 0;
            xk = 0;
            cursor_next<BN>(p, xc);
            xrow = xc.row0 + xc.mt * BN + xhalf;
          }
          progress = true;
        }
        // nothing to issue: back off briefly instead of taking issue slots
        // from the dequantiser warps of this sub-partition
        if (!progress) __nanosleep(128);
        if (!progress && (++spin & 63u) == 0) {
          if (*abort_flag) break;
          if (global_timer_ns() - t0 > p.timeout_ns) {
            fail();
            break;
          }
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA can exit
        const int32_t wfirst = wi > C::kWStages ? wi - C::kWStages : 0;
        for (int32_t j = wfirst; j < wi; ++j)
          mbar_wait_bounded(smem_u32(&wfull[j % C::kWStages]), (j / C::kWStages) & 1,
                            p.timeout_ns, nullptr);
        const int32_t xfirst = xi > C::kXStages ? xi - C::kXStages : 0;
        for (int32_t j = xfirst; j < xi; ++j)
          mbar_wait_bounded(smem_u32(&xfull[j % C::kXStages]), (j / C::kXStages) & 1,
                            p.timeout_ns, nullptr);
      }
    }
  } else if (PAIR && warp == kMmaWarp && rank != 0) {
    // ------------------------------------- activation forwarder (odd CTA)
    // The even CTA's thread issues the pair's MMAs, which read this CTA's
    // half of every activation stage: tell it when each half has landed.
    const int32_t nu = static_cast<int32_t>(u1 - u0);
    int st = 0;
    uint32_t ph = 0;
    for (int32_t i = 0; i < nu; ++i) {
      if (!PETIT_CHECK(st >= 0 && st < C::kXStages)) break;
      if (!wait_warp(&xfull[st], ph)) break;
      if (elect_one()) mbar_arrive_remote(mapa_shared(smem_u32(&xpeer[st]), 0));
      __syncwarp();
      if (++st == C::kXStages) {
        st = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == kMmaWarp || warp > C::kMmaWarpX) {
    // ------------------------------------------------------------ MMA issue
    // (CTA pairs: only the even CTA issues; each MMA covers both CTAs'
    // weight tiles, M = 256, and its completion is signalled to both CTAs)
    const int t = warp == kMmaWarp ? 0 : warp - C::kMmaWarpX;   // issues units i % kMmaThreads == t
    // The whole warp runs the loop, so every operand of tcgen05.mma is
    // warp-uniform and can stay in uniform registers; one elected lane
    // issues the MMAs and commits.  (Issued from a lone lane-0 branch each
    // MMA cost ~65 cycles of issue, which set the pace of the MMA chain.)
    {
      auto uwait = [&](uint64_t* bar, uint32_t parity) { return wait_warp(bar, parity); };

      // Segments (the CTA's units inside one tile) in order; inside a
      // segment only this issuer's units i = t, t + kMmaThreads, ...
      // (CTA-local), whose activation stage, A-buffer and phases advance by
      // kMmaThreads (a divisor of kXStages and kNumA).  32-bit counters: a
      // CTA has fewer than 2^31 units.
      const int32_t nu = static_cast<int32_t>(u1 - u0);
      const int32_t ks = static_cast<int32_t>(KS);
      const int32_t ku0 = static_cast<int32_t>(u0 - (u0 / KS) * KS);
      int32_t seg = 0;
      int32_t i = t;
      int st = t, b = t;   // t < kMmaThreads <= kNumA <= kXStages
      uint32_t ph = 0, pb = 0;
      bool ok = true;
      for (int32_t s0 = 0; s0 < nu && ok;) {
        const int32_t s1 = min(nu, s0 + (ks - (ku0 + s0) % ks));   // next tile boundary
        const int d = seg % C::kNumD;
        // Every issuer waits here, owning a unit of the segment or not: its
        // dfull arrival for this segment then cannot overtake the other
        // issuer's arrival for the segment that last used accumulator d.
        if (!uwait(&dempty[d], static_cast<uint32_t>(((seg / C::kNumD) & 1) ^ 1))) break;
        bool seg_started = false;   // this issuer has written its accumulator in this segment
        for (; i < s1; i += C::kMmaThreads) {
          if (!uwait(&xfull[st], ph) || (PAIR && !uwait(&xpeer[st], ph)) ||
              !uwait(&afull[b], pb)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!PETIT_CHECK(st >= 0 && st < C::kXStages && b >= 0 && b < C::kNumA && d >= 0 &&
                           d < C::kNumD)) {
            ok = false;
            break;
          }
          const uint32_t a_smem = smem_u32(sm_a + st * C::kABytes);
          const uint32_t d_tmem = tmem + C::kDColBase + (t * C::kNumD + d) * BN;
          const uint32_t a_tmem = tmem + b * C::kAColsPerUnit;
          if (elect_one()) {
#pragma unroll
            for (int j = 0; j < KU * (kStageK / 16); ++j) {
              // K16 step j: slab j / 4 of A, 32-byte offset inside its swizzled rows
              const uint64_t bdesc = smem_desc_kmajor_sw128(a_smem + (j >> 2) * C::kAHalfBytes) +
                                     (((j & 3) * 32) >> 4);
              if constexpr (PAIR)
                mma_ts_f16_pair(d_tmem, a_tmem + j * 8, bdesc, C::kIdesc,
                                (!seg_started && j == 0) ? 0u : 1u);
              else
                mma_ts_f16(d_tmem, a_tmem + j * 8, bdesc, C::kIdesc,
                           (!seg_started && j == 0) ? 0u : 1u);
            }
            if constexpr (PAIR) {
              mma_commit_pair(smem_u32(&mdone[st]));
              mma_commit_pair(mapa_shared(smem_u32(&mdone[st]), 1));
            } else {
              mma_commit(smem_u32(&mdone[st]));
            }
          }
          __syncwarp();
          seg_started = true;
          st += C::kMmaThreads;
          if (st >= C::kXStages) {
            st -= C::kXStages;
            ph ^= 1u;
          }
          b += C::kMmaThreads;
          if (b >= C::kNumA) {
            b -= C::kNumA;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        // every issuer arrives once per segment, when its MMAs are done
        if (elect_one()) {
          if constexpr (PAIR) {
            mma_commit_pair(smem_u32(&dfull[d]));
            mma_commit_pair(mapa_shared(smem_u32(&dfull[d]), 1));
          } else {
            mma_commit(smem_u32(&dfull[d]));
          }
        }
        __syncwarp();
        ++seg;
        s0 = s1;
      }
      // all issued MMAs complete before tensor memory is released
      if (elect_one()) {
        if constexpr (PAIR) mma_commit_pair(smem_u32(&fin[t]));
        else mma_commit(smem_u32(&fin[t]));
      }
      __syncwarp();
      mbar_wait_bounded(smem_u32(&fin[t]), 0, p.timeout_ns, nullptr);
    }
  } else if (warp < kDeqWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const int epi_tid = threadIdx.x - kEpiWarp0 * 32;
    int64_t seg = 0;
    const int64_t first_tile_of_cta = u0 / KS;
    if (warp == kEpiWarp0 && lane == 0) {
      // The first ring of weight chunks, before the grid dependency wait
      // (every stage starts free).  Issuing a bulk copy takes a while, so
      // this idle thread does it and the producer reaches the dependency
      // wait, and the activation copies after it, without delay.
      WeightStream<FMT, BN, KU> ws;
      ws.init(p, tile0_32, ku0_32, ks32, smem_u32(sm_w), smem_u32(&wfull[0]), C::kWStages, wmul,
              static_cast<int32_t>(rank));
      const uint64_t policy = p.weights_reused ? l2_policy_evict_normal() : l2_policy_evict_first();
      for (int64_t j = 0; j < u1 - u0 && j < C::kWStages; ++j) {
        if (PETIT_CHECK(ws.in_bounds(p))) ws.issue(p, policy);
        else ws.skip(p);   // every first-ring stage completes: the producer counts them
      }
      // The CTAs with the highest indices take their SMs last (as the
      // previous kernel's CTAs leave them); a CTA of the lower half pulls the
      // first ring of weight chunks of its partner in the upper half into
      // L2, so that partner's first copies hit L2.
      const int32_t half = (p.num_ctas + 1) / 2;
      if (cta + half < p.num_ctas) {
        const int32_t pc = static_cast<int32_t>(cta) + half;
        const int32_t pu0 = cta_lo(p, pc), pn = cta_lo(p, pc + 1) - pu0;
        WeightStream<FMT, BN, KU> pw;
        pw.init(p, pu0 / ks32, pu0 % ks32, ks32, 0, 0, C::kWStages, wmul,
                static_cast<int32_t>(rank));
        for (int32_t j = 0; j < pn && j < C::kWStages; ++j) {
          if (!PETIT_CHECK(pw.in_bounds(p))) break;
          bulk_prefetch_l2(pw.src, WeightStream<FMT, BN, KU>::kBytes);
          pw.advance(p);
        }
      }
    }
    // C, the partials and the counters may be in use by the previous kernel
    // on the stream until it has completed
    grid_dependency_wait();
    // epilogue factor: a device-resident global scale is read here, after the
    // grid dependency wait, so a preceding kernel may have produced it
    const float alpha_dev = p.alpha_dev ? p.alpha_scale * *p.alpha_dev : 0.0f;
    TileCursor ec = cursor_at<BN>(p, first_tile_of_cta);   // advances one tile per segment
    uint32_t epi_phase = 0;
    // bounded barrier among the four epilogue warps (a hardware named
    // barrier has no time limit)
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(epi_bar));
      const bool ok = wait_lane(epi_bar, epi_phase & 1u);
      ++epi_phase;
      return ok;
    };
    // 128/256-row tiles: 16 rows (row0 .. row0 + 15 of group g's output,
    // columns col0 + 0..127) from the four epilogue warps, each holding its
    // 32 columns, are staged in shared memory and written as whole 256-byte
    // row segments, a 16-byte vector per lane.  Stored directly, each warp's
    // 64-byte piece of each row took ~5x as long (measured on GB300: 10 us
    // against 2 us to drain a 256-row tile of the gate_up projection).
    auto put_rows = [&](const float (&val)[16], uint16_t* c_g, int64_t row0, int64_t col0,
                        int64_t g_rows, float alpha) {
      if constexpr (C::kStageC > 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) stage_c[j * kTileN + r] = out_bits<FMT>(alpha * val[j]);
        if (!epi_sync()) return false;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int row = 4 * q + 2 * s2 + (lane >> 4);   // warp q writes rows 4q .. 4q + 3
          const int col = (lane & 15) * 8;
          const int64_t mrow = row0 + row;
          if (mrow < g_rows &&
              PETIT_CHECK(col0 + col + 8 <= p.n &&
                          (c_g - p.c) + mrow * p.n + col0 + col + 8 <= p.chk_c_elems))
            *reinterpret_cast<uint4*>(c_g + mrow * p.n + col0 + col) =
                *reinterpret_cast<const uint4*>(stage_c + row * kTileN + col);
        }
        return epi_sync();   // before the buffer is written again
      } else {
        return false;
      }
    };
    for (int64_t u = u0; u < u1; ++seg) {
      const int64_t tile = u / KS;
      const int64_t seg_end = (tile + 1) * KS < u1 ? (tile + 1) * KS : u1;
      const bool full_tile = (u == tile * KS) && (seg_end == (tile + 1) * KS);
      const int64_t nt = ec.nt, mt = ec.mt;
      const int64_t g_rows = p.row_off[ec.g + 1] - p.row_off[ec.g];  // this group's activation rows
      uint16_t* const c_g = p.c + static_cast<int64_t>(p.row_off[ec.g]) * p.n;
      const float alpha = p.alpha_dev ? alpha_dev : p.group_alpha[ec.g];
      cursor_next<BN>(p, ec);
      const int d = static_cast<int>(seg % C::kNumD);
      // split tile: its contributors and their partial slots (every
      // contributor but the first starts inside the tile, slot 2c; the first
      // uses its second slot unless its range starts at the tile)
      int64_t c_first = 0, c_last = 0, first_slot = 0;
      uint32_t* ctr = nullptr;
      const bool last_seg = seg_end == u1;
      bool early = false;   // every other contributor has arrived: sum now
      if (!full_tile) {
        c_first = cta_of_unit(p, tile * KS);
        c_last = cta_of_unit(p, (tile + 1) * KS - 1);
        first_slot =
            2 * sid(c_first) + (cta_lo(p, static_cast<int32_t>(c_first)) / KS == tile ? 0 : 1);
        if (!PETIT_CHECK(c_first >= 0 && c_first <= c_last && c_last < P &&
                         sid(c_first) < kMaxCtas && first_slot >= 0 && first_slot < 2 * NS))
          break;
        ctr = &p.counters[sid(c_first)];
        // first look while the segment's MMAs run
        if (last_seg && epi_tid == 0)
          *epi_flag = ld_acquire_gpu(ctr) == static_cast<uint32_t>(c_last - c_first);
      }
      if (!PETIT_CHECK(d >= 0 && d < C::kNumD)) break;
      if (!wait_lane(&dfull[d], static_cast<uint32_t>((seg / C::kNumD) & 1))) break;
      tc_fence_after();
      // issuer t wrote its accumulator iff the segment holds a unit with
      // CTA-local index i % kMmaThreads == t
      const int seg_len = static_cast<int>(seg_end - u);
      const int seg_r0 = static_cast<int>((u - u0) % C::kMmaThreads);
      uint32_t has = 0;   // bit t: issuer t contributed
#pragma unroll
      for (int t = 0; t < C::kMmaThreads; ++t)
        if ((t - seg_r0 + C::kMmaThreads) % C::kMmaThreads < seg_len) has |= 1u << t;
      if (!full_tile && last_seg) {
        // second look once the MMAs are done
        if (epi_tid == 0 && !*epi_flag)
          *epi_flag = ld_acquire_gpu(ctr) == static_cast<uint32_t>(c_last - c_first);
        if (!epi_sync()) break;
        early = *epi_flag != 0;
        if (early) {
          // the CTA's last segment, summed by all warps after the final
          // barrier from the accumulator that stays in tensor memory
          if (epi_tid == 0) {
            atomicExch(ctr, 0u);   // no other contributor touches it again
            fix->c_g = c_g;
            fix->c_first = c_first;
            fix->c_last = c_last;
            fix->first_slot = first_slot;
            fix->row0 = static_cast<int64_t>(mt) * BN;
            fix->col0 = (static_cast<int64_t>(nt) * wmul + rank) * kTileN;
            fix->g_rows = g_rows;
            fix->alpha = alpha;
            fix->d = d;
            fix->has = has;
            fix->valid = 1;
          }
          u = seg_end;
          continue;
        }
      }
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(32 * q) << 16) + C::kDColBase + d * BN;
      const int64_t ncol = (static_cast<int64_t>(nt) * wmul + rank) * kTileN + r;
      const int64_t slot = 2 * sid(cta) + (tile == first_tile_of_cta ? 0 : 1);
      float* my_slot = p.partials + static_cast<size_t>(slot) * (BN * kTileN);
      // (a partial slot holds BN x 128 floats; r < 128)
      if (!full_tile && !PETIT_CHECK(slot >= 0 && slot < 2 * NS)) break;
      bool c_ok = true;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        // the contributing accumulators, added in issuer order
        uint32_t v[16];
        bool have = false;
#pragma unroll
        for (int t = 0; t < C::kMmaThreads; ++t) {
          if (has & (1u << t)) {
            uint32_t w[16];
            tmem_ld_x16(tbase + (t * C::kNumD) * BN + c0, w);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              v[j] = have ? __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(w[j])) : w[j];
            have = true;
          }
        }
        if (full_tile && C::kStageC > 0) {
          float fv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) fv[j] = __uint_as_float(v[j]);
          if (!put_rows(fv, c_g, static_cast<int64_t>(mt) * BN + c0, ncol - r, g_rows, alpha)) {
            c_ok = false;
            break;
          }
        } else if (full_tile) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t mrow = static_cast<int64_t>(mt) * BN + c0 + j;
            if (mrow < g_rows && PETIT_CHECK(ncol < p.n && (c_g - p.c) + mrow * p.n + ncol <
                                                             p.chk_c_elems))
              c_g[mrow * p.n + ncol] = out_bits<FMT>(alpha * __uint_as_float(v[j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) my_slot[(c0 + j) * kTileN + r] = __uint_as_float(v[j]);
        }
      }
      if (!c_ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // (CTA pairs: the even CTA's issuer waits for both CTAs' epilogues)
        if (PAIR && rank != 0) mbar_arrive_remote(mapa_shared(smem_u32(&dempty[d]), 0));
        else mbar_arrive(smem_u32(&dempty[d]));
      }
      if (!full_tile) {
        // Ordering without per-thread fences: the group barrier (mbarrier
        // arrive = release, wait = acquire, CTA scope) orders every epilogue
        // thread's partial stores before thread 0's GPU-scope acq_rel
        // arrival, which releases them cumulatively to the CTA that acquires
        // the counter last; that CTA's acquire reaches its other epilogue
        // threads through its own group barrier before their loads.
        if (!epi_sync()) break;
        if (epi_tid == 0) {
          const uint32_t old = atomic_add_acq_rel_gpu(ctr, 1u);
          const int is_last = (static_cast<int64_t>(old) == c_last - c_first);
          if (is_last) atomicExch(ctr, 0u);  // ready for the next call
          *epi_flag = is_last;
        }
        if (!epi_sync()) break;
        if (*epi_flag && last_seg) {
          // the CTA's last segment: summed by all warps after the final barrier
          if (epi_tid == 0) {
            fix->c_g = c_g;
            fix->c_first = c_first;
            fix->c_last = c_last;
            fix->first_slot = first_slot;
            fix->row0 = static_cast<int64_t>(mt) * BN;
            fix->col0 = (static_cast<int64_t>(nt) * wmul + rank) * kTileN;
            fix->g_rows = g_rows;
            fix->alpha = alpha;
            fix->d = d;
            fix->has = has;
            fix->valid = 1;
          }
        } else if (*epi_flag) {
          // contributors' partials are summed in CTA order (deterministic);
          // loads are batched (kFixBatch contributors x 16 columns in flight),
          // so the reduction costs a few L2 round trips, not one per value
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
#pragma unroll 1
            for (int64_t cb = c_first; cb <= c_last; cb += kFixBatch) {
              float tv[kFixBatch][16];
#pragma unroll
              for (int x = 0; x < kFixBatch; ++x) {
                const int64_t c = cb + x;
                if (c <= c_last) {
                  const int64_t cs = c == c_first ? first_slot : 2 * sid(c);
                  if (!PETIT_CHECK(cs >= 0 && cs < 2 * NS)) continue;
                  const float* src =
                      p.partials + static_cast<size_t>(cs) * (BN * kTileN) + c0 * kTileN + r;
#pragma unroll
                  for (int j = 0; j < 16; ++j) tv[x][j] = __ldcg(src + j * kTileN);
                }
              }
#pragma unroll
              for (int x = 0; x < kFixBatch; ++x) {
                if (cb + x <= c_last) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) acc[j] += tv[x][j];
                }
              }
            }
            // (stored directly: here the partial loads set the pace, and
            // staging, with its barriers between the warps, was slower)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int64_t mrow = static_cast<int64_t>(mt) * BN + c0 + j;
              if (mrow < g_rows && PETIT_CHECK(ncol < p.n && (c_g - p.c) + mrow * p.n + ncol <
                                                               p.chk_c_elems))
                c_g[mrow * p.n + ncol] = out_bits<FMT>(alpha * acc[j]);
            }
          }
        }
        if (!epi_sync()) break;
      }
      u = seg_end;
    }
  } else {
    // ---------------------------------------------------------- dequantise
    // kDeqGroups groups of four warps take units round-robin; a warp decodes
    // both 64-k halves of its 32 rows, one 32-k group pair at a time.  The
    // dequantiser warps of an SM sub-partition then work on different
    // units, so one's barrier waits and round trips overlap the others'
    // decode arithmetic.  Only shared and tensor memory are touched, so the
    // first units are dequantised before the previous kernel has finished.
    const int grp = (warp - kDeqWarp0) / kDeqGroupWarps;
    const int q = warp & 3;         // tensor-memory lane quarter
    const int r = 32 * q + lane;    // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    constexpr int G = C::kDeqGroups;
    // this group's units i = grp, grp + G, ... (CTA-local); the weight
    // stage, A-buffer and the activation stage of unit i - kNumA advance by
    // G and wrap (G <= kNumA <= kXStages, G <= kWStages)
    const int32_t nu = static_cast<int32_t>(u1 - u0);
    int st = grp, b = grp;
    uint32_t ph = 0;
    // first own unit that reuses an A-buffer: i0 >= kNumA, i0 = grp (mod G)
    constexpr int kFirstReuse0 = (C::kNumA + G - 1) / G * G;   // for grp = 0
    const int i0 = kFirstReuse0 + grp - (kFirstReuse0 - G + grp >= C::kNumA ? G : 0);
    int st2 = (i0 - C::kNumA) % C::kXStages;
    uint32_t ph2 = ((i0 - C::kNumA) / C::kXStages) & 1;
    for (int32_t i = grp; i < nu; i += G) {
      if (!PETIT_CHECK(st >= 0 && st < C::kWStages && b >= 0 && b < C::kNumA && st2 >= 0 &&
                       st2 < C::kXStages))
        break;
      if (!wait_lane(&wfull[st], ph)) break;
      bool ok = true;
      if constexpr (FMT == kMXFP4) {
        // The repack's per-chunk flag bytes (warp-uniform), read once per
        // unit: the unit's decode takes one multiply per word when every
        // scale code of its chunks is <= 128 (both variants of the loop are
        // compiled; a flag test inside the unrolled loop cost 5 % of the
        // MXFP4 decode step).
        bool fast = true;
#pragma unroll
        for (int j = 0; j < KU; ++j)
          fast = fast &&
                 sm_w[st * C::kWBytes + j * T::kChunkBytes + kWChunkBytes + T::kSChunkBytes];
        auto unit = [&](auto fast_tag) {
          constexpr bool kFast = decltype(fast_tag)::value;
#pragma unroll
          for (int hj = 0; hj < 2 * KU; ++hj) {
            const int h = hj / KU, j = hj % KU;
            const uint8_t* chunk = sm_w + st * C::kWBytes + j * T::kChunkBytes;
            const uint4 g0 =
                *reinterpret_cast<const uint4*>(chunk + ((2 * h) * kTileN + r) * 16);
            const uint4 g1 =
                *reinterpret_cast<const uint4*>(chunk + ((2 * h + 1) * kTileN + r) * 16);
            uint32_t o[2][16];
            const uint32_t sv =
                *reinterpret_cast<const uint16_t*>(chunk + kWChunkBytes + (h * kTileN + r) * 2);
            decode_group<FMT, kFast>(g0, sv & 0xFFu, o[0]);
            decode_group<FMT, kFast>(g1, (sv >> 8) & 0xFFu, o[1]);
            if (hj == 2 * KU - 1) {
              // the decode consumed every byte this warp read: release the chunk
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&wfree[st]));
            }
            if (hj == 0 && i >= C::kNumA) {
              // A-buffer b was last used by unit i - kNumA: wait for its
              // MMAs, and order the stores below after their operand reads
              if (!wait_lane(&mdone[st2], ph2)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t acol =
                tmem + lane_base + b * C::kAColsPerUnit + j * (kStageK / 2) + (2 * h) * 16;
            tmem_st_x16(acol, o[0]);
            tmem_st_x16(acol + 16, o[1]);
          }
        };
        if (fast) unit(std::true_type{});
        else unit(std::false_type{});
      } else {
#pragma unroll
        for (int hj = 0; hj < 2 * KU; ++hj) {
          const int h = hj / KU, j = hj % KU;
          const uint8_t* chunk = sm_w + st * C::kWBytes + j * T::kChunkBytes;
          const uint4 g0 = *reinterpret_cast<const uint4*>(chunk + ((2 * h) * kTileN + r) * 16);
          const uint4 g1 =
              *reinterpret_cast<const uint4*>(chunk + ((2 * h + 1) * kTileN + r) * 16);
          uint32_t o[2][16];
          const uint32_t sv =
              *reinterpret_cast<const uint32_t*>(chunk + kWChunkBytes + (h * kTileN + r) * 4);
          decode_group<FMT>(g0, sv & 0xFFFFu, o[0]);
          decode_group<FMT>(g1, sv >> 16, o[1]);
          if (hj == 2 * KU - 1) {
            // the decode consumed every byte this warp read: release the chunk
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&wfree[st]));
          }
          if (hj == 0 && i >= C::kNumA) {
            // A-buffer b was last used by unit i - kNumA: wait for its MMAs,
            // and order the stores below after their operand reads
            if (!wait_lane(&mdone[st2], ph2)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t acol =
              tmem + lane_base + b * C::kAColsPerUnit + j * (kStageK / 2) + (2 * h) * 16;
          tmem_st_x16(acol, o[0]);
          tmem_st_x16(acol + 16, o[1]);
        }
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // (CTA pairs: the even CTA's MMA reads both CTAs' A-buffers)
        if (PAIR && rank != 0) mbar_arrive_remote(mapa_shared(smem_u32(&afull[b]), 0));
        else mbar_arrive(smem_u32(&afull[b]));
      }
      st += G;
      if (st >= C::kWStages) {
        st -= C::kWStages;
        ph ^= 1u;
      }
      b += G;
      if (b >= C::kNumA) b -= C::kNumA;
      if (i >= C::kNumA) {
        st2 += G;
        if (st2 >= C::kXStages) {
          st2 -= C::kXStages;
          ph2 ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Deferred sum of the last segment's split tile (see FixJob), by the
  // warps of kFixGroups groups of four (one warp per tensor-memory lane
  // quarter), each group taking BN / kFixGroups activation rows: a thread
  // owns one weight row r, reads this CTA's accumulator for its rows from
  // tensor memory and the other contributors' partials (consecutive threads
  // at consecutive addresses), adds them in CTA order and writes C.  The
  // epilogue's acquire of the arrival counter reaches every thread through
  // the barrier above.
  if constexpr (C::kStageC > 0) {
    // 128/256-row tiles: the same sum, written through a shared-memory stage
    // in 256-byte row segments (as the epilogue writes whole tiles); the
    // activation ring is free by now and holds one 16-row stage per group.
    // Every warp runs the same loop, so the CTA-wide barriers match; the
    // decision to run it is read by all threads before any check below can
    // raise the abort flag.
    const bool run_fix = fix->valid && !*abort_flag;
    __syncthreads();
    if (run_fix) {
      const FixJob f = *fix;
      constexpr int kFixGroups = C::kThreads / 32 >= 16 ? 4 : 2;
      constexpr int kCols = BN / kFixGroups;   // activation rows per group (>= 32)
      const int fg = warp >> 2;
      const bool mine =
          fg < kFixGroups &&
          PETIT_CHECK(f.d >= 0 && f.d < C::kNumD && f.c_first >= 0 && f.c_first <= cta &&
                      cta <= f.c_last && f.c_last < P && f.first_slot >= 0 &&
                      f.first_slot < 2 * NS);
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::kDColBase +
                             f.d * BN + fg * kCols;
      uint16_t* gst = reinterpret_cast<uint16_t*>(sm_a) + (fg % kFixGroups) * 16 * kTileN;
#pragma unroll 1
      for (int c0 = 0; c0 < kCols; c0 += 16) {
        const int m0 = fg * kCols + c0;   // first activation row (tile-local)
        if (mine) {
          float own[16];
          bool have = false;
#pragma unroll
          for (int t = 0; t < C::kMmaThreads; ++t) {
            if (f.has & (1u << t)) {
              uint32_t x[16];
              tmem_ld_x16(tbase + (t * C::kNumD) * BN + c0, x);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j)
                own[j] = have ? own[j] + __uint_as_float(x[j]) : __uint_as_float(x[j]);
              have = true;
            }
          }
          float acc[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
#pragma unroll 1
          for (int64_t cb = f.c_first; cb <= f.c_last; cb += kFixBatch) {
            float tv[kFixBatch][16];
#pragma unroll
            for (int x = 0; x < kFixBatch; ++x) {
              const int64_t c = cb + x;
              if (c <= f.c_last && c != cta) {
                const float* src =
                    p.partials +
                    static_cast<size_t>(c == f.c_first ? f.first_slot : 2 * sid(c)) *
                        (BN * kTileN) +
                    m0 * kTileN + r;
#pragma unroll
                for (int j = 0; j < 16; ++j) tv[x][j] = __ldcg(src + j * kTileN);
              }
            }
#pragma unroll
            for (int x = 0; x < kFixBatch; ++x) {
              const int64_t c = cb + x;
              if (c <= f.c_last) {
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] += c == cta ? own[j] : tv[x][j];
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) gst[j * kTileN + r] = out_bits<FMT>(f.alpha * acc[j]);
        }
        __syncthreads();
        if (mine) {
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            const int row = 4 * q + 2 * s2 + (lane >> 4);   // warp q writes rows 4q .. 4q + 3
            const int col = (lane & 15) * 8;
            const int64_t mrow = f.row0 + m0 + row;
            if (mrow < f.g_rows &&
                PETIT_CHECK(f.col0 + col + 8 <= p.n &&
                            (f.c_g - p.c) + mrow * p.n + f.col0 + col + 8 <= p.chk_c_elems))
              *reinterpret_cast<uint4*>(f.c_g + mrow * p.n + f.col0 + col) =
                  *reinterpret_cast<const uint4*>(gst + row * kTileN + col);
          }
        }
        __syncthreads();
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  } else {
    if (fix->valid && !*abort_flag) {
      const FixJob f = *fix;
      constexpr int kFixGroups = C::kThreads / 32 >= 16 ? 4 : 2;
      constexpr int kCols = BN / kFixGroups;               // activation rows per group
      constexpr int kLd = kCols >= 16 ? 16 : 4;            // columns per tensor-memory load
      const int fg = warp >> 2;
      if (fg < kFixGroups && !*abort_flag &&
          PETIT_CHECK(f.d >= 0 && f.d < C::kNumD && f.c_first >= 0 && f.c_first <= cta &&
                      cta <= f.c_last && f.c_last < P && f.first_slot >= 0 &&
                      f.first_slot < 2 * NS)) {
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::kDColBase +
                               f.d * BN + fg * kCols;
  #pragma unroll 1
        for (int c0 = 0; c0 < kCols; c0 += kLd) {
          float own[kLd];
  #pragma unroll
          for (int j = 0; j < kLd; ++j) own[j] = 0.0f;
          bool have = false;
  #pragma unroll
          for (int t = 0; t < C::kMmaThreads; ++t) {
            if (f.has & (1u << t)) {
              uint32_t x[kLd];
              if constexpr (kLd == 16) {
                tmem_ld_x16(tbase + (t * C::kNumD) * BN + c0, x);
              } else {
                tmem_ld_x4(tbase + (t * C::kNumD) * BN + c0, x);
              }
              tmem_wait_ld();
  #pragma unroll
              for (int j = 0; j < kLd; ++j) own[j] = have ? own[j] + __uint_as_float(x[j]) : __uint_as_float(x[j]);
              have = true;
            }
          }
          const int m0 = fg * kCols + c0;   // first activation row (tile-local)
          float acc[kLd];
  #pragma unroll
          for (int j = 0; j < kLd; ++j) acc[j] = 0.0f;
  #pragma unroll 1
          for (int64_t cb = f.c_first; cb <= f.c_last; cb += kFixBatch) {
            float tv[kFixBatch][kLd];
  #pragma unroll
            for (int x = 0; x < kFixBatch; ++x) {
              const int64_t c = cb + x;
              if (c <= f.c_last && c != cta) {
                const float* src = p.partials +
                                   static_cast<size_t>(c == f.c_first ? f.first_slot : 2 * sid(c)) *
                                       (BN * kTileN) +
                                   m0 * kTileN + r;
  #pragma unroll
                for (int j = 0; j < kLd; ++j) tv[x][j] = __ldcg(src + j * kTileN);
              }
            }
  #pragma unroll
            for (int x = 0; x < kFixBatch; ++x) {
              const int64_t c = cb + x;
              if (c <= f.c_last) {
  #pragma unroll
                for (int j = 0; j < kLd; ++j) acc[j] += c == cta ? own[j] : tv[x][j];
              }
            }
          }
  #pragma unroll
          for (int j = 0; j < kLd; ++j) {
            const int64_t mrow = f.row0 + m0 + j;
            if (mrow < f.g_rows &&
                PETIT_CHECK(f.col0 + r < p.n &&
                            (f.c_g - p.c) + mrow * p.n + f.col0 + r < p.chk_c_elems))
              f.c_g[mrow * p.n + f.col0 + r] = out_bits<FMT>(f.alpha * acc[j]);
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }
  if constexpr (PAIR) {
    // Neither CTA of a pair frees its tensor memory or exits while the
    // other may still use it: the even CTA's MMAs (all complete once its
    // issuer's final commit has been waited on) read and write both CTAs'
    // tensor memory and read the odd CTA's shared memory, and each CTA
    // arrives on the other's barriers.  Every thread of both CTAs gets here
    // after bounded work only.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc_pair(tmem, kTmemCols);
  } else {
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  }
  // a wait that ran out anywhere in the CTA is reported by thread 0, which
  // has passed the grid dependency wait
  if (threadIdx.x == 0 && *abort_flag)
    atomicOr(p.status, (*abort_flag & kAbortBounds) ? kStatusBounds : kStatusTimeout);
}

template <int FMT, int BN, int KU, bool PAIR = false>
cudaError_t launch_t(const Params& prm, const CUtensorMap& tmap, cudaStream_t stream, int dev) {
  using C = Cfg<FMT, BN, KU, PAIR>;
  // the dynamic shared-memory limit is raised once per device
  static std::atomic<bool> attr_done[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<FMT, BN, KU, PAIR>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  // CTA pairs: two CTAs (a cluster) per work range
  cfg.gridDim = dim3(static_cast<unsigned>(prm.num_ctas * (PAIR ? 2 : 1)));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<FMT, BN, KU, PAIR>, prm, tmap);
}

// How many CTA pairs of the pair kernel (this format and tile height) can be
// resident at once on the current device; 0 if the query fails.
template <int FMT, int BN>
int pair_capacity_t() {
  using C = Cfg<FMT, BN, 1, true>;
  auto kern = gemm_kernel<FMT, BN, 1, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxBoundCtas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int FMT>
cudaError_t launch_fmt(int bn, int ku, bool pair, const Params& prm, const CUtensorMap& tmap,
                       cudaStream_t s, int dev) {
  if (pair) {
    if (ku != 1) return cudaErrorInvalidValue;
    switch (bn) {
      case 128: return launch_t<FMT, 128, 1, true>(prm, tmap, s, dev);
      case 256: return launch_t<FMT, 256, 1, true>(prm, tmap, s, dev);
      default: return cudaErrorInvalidValue;
    }
  }
  if (ku == 2) {
    switch (bn) {
      case 16: return launch_t<FMT, 16, 2>(prm, tmap, s, dev);
      case 32: return launch_t<FMT, 32, 2>(prm, tmap, s, dev);
      case 64: return launch_t<FMT, 64, 2>(prm, tmap, s, dev);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_t<FMT, 16, 1>(prm, tmap, s, dev);
    case 32: return launch_t<FMT, 32, 1>(prm, tmap, s, dev);
    case 64: return launch_t<FMT, 64, 1>(prm, tmap, s, dev);
    case 128: return launch_t<FMT, 128, 1>(prm, tmap, s, dev);
    case 256: return launch_t<FMT, 256, 1>(prm, tmap, s, dev);
    default: return cudaErrorInvalidValue;
  }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Stream-K ranges.  The CTAs of a launch take their SMs in index order as
// the previous kernel's CTAs leave them, so under back-to-back launches the
// last few indices start last -- measured on GB300 for the decode step, the
// last four CTAs finish their MMAs ~1.5-2.5 us after the median one and the
// lateness halves about every seven indices below them.  With equal ranges
// they set the end of every kernel, so their ranges shrink:
//   deficit(c) = kLateStartNs * exp((c - (P - 1)) / (P / 15)) / unit time
// units for CTA c, and every CTA shares the total back.
constexpr double kLateStartNs = 1600.0;

void plan_bounds(GemmPlan& pl, double late_ns) {
  const int P = pl.num_ctas;
  const int64_t U = pl.units;
  pl.use_bounds = false;
  // measured on GB300: 1 % off the m = 16 decode step; with 128/256-row
  // tiles (prefill) the skew was 1 % slower, so those keep the even split
  if (P < 16 || P > kMaxBoundCtas || late_ns <= 0.0 || pl.bn > 64) return;
  // rough time of one unit on one SM at the decode pace (its weight bytes
  // at the SM's share of HBM bandwidth)
  const double unit_ns = 240.0 * pl.ku;
  const double tau = P / 15.0;
  double deficit[kMaxBoundCtas], total = 0.0;
  for (int c = 0; c < P; ++c) {
    deficit[c] = late_ns / unit_ns * std::exp((c - (P - 1)) / tau);
    total += deficit[c];
  }
  const double base = (static_cast<double>(U) + total) / P;
  double share[kMaxBoundCtas], sum = 0.0;
  for (int c = 0; c < P; ++c) {
    share[c] = std::max(base - deficit[c], std::max(1.0, 0.5 * base));
    sum += share[c];
  }
  double cum = 0.0;
  pl.bound[0] = 0;
  for (int c = 1; c < P; ++c) {
    cum += share[c - 1] * static_cast<double>(U) / sum;
    int64_t b = std::llround(cum);
    b = std::max<int64_t>(b, pl.bound[c - 1] + 1);   // every CTA keeps a unit
    b = std::min<int64_t>(b, U - (P - c));
    pl.bound[c] = static_cast<int32_t>(b);
  }
  pl.bound[P] = static_cast<int32_t>(U);
  pl.use_bounds = true;
}

std::atomic<int> g_tile_override{0};   // bn | ku << 16, or 0: the planner decides
std::atomic<int> g_pair_mode{0};       // 0: CTA pairs where they pay, 1: never, 2: wherever possible
// bounds-checking build: extents the checks use in place of the true ones
// (negative: the true extent)
std::atomic<int64_t> g_check_weight_bytes{-1};
std::atomic<int64_t> g_check_c_elems{-1};

double late_start_ns() { return kLateStartNs; }

}  // namespace

int tile_override() { return g_tile_override.load(std::memory_order_relaxed); }

bool set_pair_mode(int mode) {
  if (mode < 0 || mode > 2) return false;
  g_pair_mode.store(mode);
  return true;
}

int pair_capacity() {
  int cap = 1 << 30;
  for (const int c : {pair_capacity_t<kNVFP4, 128>(), pair_capacity_t<kNVFP4, 256>(),
                      pair_capacity_t<kMXFP4, 128>(), pair_capacity_t<kMXFP4, 256>(),
                      pair_capacity_t<kNVFP4F16, 128>(), pair_capacity_t<kNVFP4F16, 256>()})
    cap = std::min(cap, c);
  return std::min(cap, kMaxBoundCtas);
}

bool bounds_checking() {
#ifdef PETIT_CHECK_BOUNDS
  return true;
#else
  return false;
#endif
}

bool set_check_limits(int64_t weight_bytes, int64_t c_elems) {
  if (!bounds_checking()) return false;
  g_check_weight_bytes.store(weight_bytes);
  g_check_c_elems.store(c_elems);
  return true;
}

bool set_tile_override(int bn, int ku) {
  if (bn == 0 && ku == 0) {
    g_tile_override.store(0);
    return true;
  }
  if ((bn != 16 && bn != 32 && bn != 64 && bn != 128 && bn != 256) || (ku != 1 && ku != 2) ||
      (ku == 2 && bn > 64))
    return false;
  g_tile_override.store(bn | (ku << 16));
  return true;
}

GemmPlan plan_grouped(const int64_t* row_off, int num_groups, int64_t n, int64_t k, int fmt,
                      int num_sms, int pair_cap) {
  GemmPlan pl{};
  pl.fmt = fmt;
  pl.num_groups = num_groups;
  int64_t max_rows = 0;
  for (int g = 0; g < num_groups; ++g) {
    const int64_t r = row_off[g + 1] - row_off[g];
    if (r > max_rows) max_rows = r;
  }
  const int64_t m = max_rows > 0 ? max_rows : 1;
  pl.bn = m <= 16 ? 16 : (m <= 32 ? 32 : (m <= 64 ? 64 : (m <= 128 ? 128 : 256)));
  if (num_groups > 1) {
    // groups of different sizes share one tile height: take the one with the
    // least work, counting each activation tile as one pass over the group's
    // weights and an N = 256 tile as two (its MMAs, not the weight stream,
    // set its pace)
    int64_t best = -1;
    for (int bn = 16; bn <= 256; bn *= 2) {
      int64_t tiles = 0;
      for (int g = 0; g < num_groups; ++g) tiles += (row_off[g + 1] - row_off[g] + bn - 1) / bn;
      const int64_t cost = tiles * (bn > 128 ? bn / 128 : 1);
      if (best < 0 || cost < best) {
        best = cost;
        pl.bn = bn;
      }
    }
  }
  // CTA pairs (cta_group::2 MMAs over two adjacent weight tiles) for 128-
  // and 256-row tiles of a single GEMM whose n holds whole tile pairs
  const int pair_mode = g_pair_mode.load(std::memory_order_relaxed);
  const bool pair_ok = pair_cap > 0 && num_groups == 1 && n % (2 * kTileN) == 0 && pair_mode != 1;
  if (num_groups == 1 && pl.bn == 256 && m <= 256) {
    // N = 256 dequantises each weight once for all rows, but halves the
    // number of work units; small matrices keep two 128-row tiles so that
    // every CTA still has a long pipeline to amortise its fixed costs over
    const int64_t units256 = num_groups * (n / kTileN) * (k / kStageK);
    if (units256 < 48 * static_cast<int64_t>(num_sms)) pl.bn = 128;
  }
  // two chunks per unit halves the copy requests when the A tile is small
  pl.ku = (pl.bn <= 64 && (k / kStageK) % 2 == 0) ? 2 : 1;
  const int ov = tile_override();
  if (ov != 0) {
    // a forced tile shape (tuning and tests): BN as given, two chunks per
    // unit only where that kernel exists and k holds an even number of them
    pl.bn = ov & 0xFFFF;
    pl.ku = ((ov >> 16) == 2 && pl.bn <= 64 && (k / kStageK) % 2 == 0) ? 2 : 1;
  }
  // Measured on GB300 (Llama-3-70B shapes, m = 128..512): CTA pairs are
  // 5-14 % faster with 256-row tiles and on large matrices with 128-row
  // tiles (gate_up), and level with single CTAs on small 128-row-tile
  // problems (QKV, O: 27-67 pair units per range), which stay on single CTAs
  if (pair_ok && pl.bn >= 128 && pl.ku == 1) {
    const int64_t pair_units = static_cast<int64_t>(n / (2 * kTileN)) * (k / kStageK) *
                               ((m + pl.bn - 1) / pl.bn);
    pl.pair = pair_mode == 2 || pl.bn == 256 || pair_units >= 100 * static_cast<int64_t>(pair_cap);
  }
  // work tiles: 128 weight rows, or 256 (a tile pair) with CTA pairs
  pl.n_tiles = static_cast<int>(n / (kTileN * (pl.pair ? 2 : 1)));
  pl.k_stages = static_cast<int>(k / kStageK);
  int64_t tiles = 0;
  for (int g = 0; g <= num_groups; ++g) {
    pl.row_off[g] = static_cast<int32_t>(row_off[g]);
    pl.tile_base[g] = static_cast<int32_t>(tiles);
    if (g == num_groups) break;
    const int64_t mt = (row_off[g + 1] - row_off[g] + pl.bn - 1) / pl.bn;
    if (mt > 1) pl.weights_reused = true;
    tiles += mt * pl.n_tiles;
  }
  pl.units = tiles * (pl.k_stages / pl.ku);
  // work ranges: one per SM, or one per resident CTA pair
  const int64_t ranges = pl.pair ? pair_cap : num_sms;
  pl.num_ctas = static_cast<int>(pl.units < ranges ? pl.units : ranges);
  if (pl.num_ctas < 1) pl.num_ctas = 1;
  if (pl.num_ctas * (pl.pair ? 2 : 1) > kMaxCtas) pl.num_ctas = kMaxCtas / (pl.pair ? 2 : 1);
  if (!pl.pair && pl.bn == 128 && num_groups == 1) {
    // Tile-aligned ranges.  With 128-row tiles each of the two MMA issuers
    // has one accumulator, so a range that crosses a tile boundary stalls
    // its MMAs while the epilogue drains the finished tile: measured on
    // GB300 at about 15 units' time.  Where whole tiles, or equal parts of
    // them, give every CTA one segment on fewer CTAs for less total time,
    // take that (O at m = 128: 26.0 -> 23.7 us, at m = 256: 36.5 -> 35.0 us
    // on 128 CTAs; QKV, and down with its long tiles, keep every SM).
    const int64_t per_tile = pl.k_stages / pl.ku;
    auto cost = [&](int64_t P, bool aligned) {
      const double L = static_cast<double>((pl.units + P - 1) / P);
      return L + (aligned ? 0.0 : 15.0 * static_cast<double>(pl.units) / P / per_tile);
    };
    double best = cost(pl.num_ctas, false);
    for (int64_t parts = 1; parts <= 4; ++parts) {
      const int64_t P = tiles * parts;
      if (P > num_sms || per_tile % parts != 0) continue;
      const double c = cost(P, true);
      if (c < best) {
        best = c;
        pl.num_ctas = static_cast<int>(P);
      }
    }
  }
  if (pl.units < (int64_t(1) << 31)) plan_bounds(pl, late_start_ns());
  pl.ws.counters_off = kWsHeaderBytes;
  pl.ws.partials_off = align_up(kWsHeaderBytes + kWsCountersBytes, 256);
  // two partial slots per CTA (a work range has two CTAs with CTA pairs)
  pl.ws.total = pl.ws.partials_off + sizeof(float) * 2ull * static_cast<size_t>(pl.num_ctas) *
                                         (pl.pair ? 2 : 1) * pl.bn * kTileN;
  return pl;
}

GemmPlan plan_gemm(int64_t m, int64_t n, int64_t k, int fmt, int num_sms, int pair_cap) {
  const int64_t off[2] = {0, m};
  return plan_grouped(off, 1, n, k, fmt, num_sms, pair_cap);
}

cudaError_t launch_gemm(const GemmPlan& pl, const GemmArgs& a, const CUtensorMap& tmap,
                        cudaStream_t stream) {
  Params prm{};
  prm.rep = a.rep;
  prm.c = static_cast<uint16_t*>(a.C);
  prm.partials = reinterpret_cast<float*>(a.workspace + pl.ws.partials_off);
  prm.counters = reinterpret_cast<uint32_t*>(a.workspace + pl.ws.counters_off);
  prm.status = reinterpret_cast<uint32_t*>(a.workspace);
  prm.n = static_cast<int32_t>(a.n);
  prm.n_tiles = pl.n_tiles;
  prm.k_units = pl.k_stages / pl.ku;
  prm.units = pl.units;
  prm.num_ctas = pl.num_ctas;
  prm.units_q = static_cast<int32_t>(pl.units / pl.num_ctas);
  prm.units_r = static_cast<int32_t>(pl.units % pl.num_ctas);
  prm.use_bounds = pl.use_bounds ? 1 : 0;
  if (pl.use_bounds)
    for (int c = 0; c <= pl.num_ctas; ++c) prm.bound[c] = pl.bound[c];
  prm.weights_reused = pl.weights_reused ? 1 : 0;
  prm.alpha_dev = a.alpha_dev;
  prm.alpha_scale = a.alpha_scale;
  prm.timeout_ns = a.timeout_ns;
  prm.rep_stride = a.rep_stride;
  prm.num_groups = pl.num_groups;
  for (int g = 0; g <= pl.num_groups; ++g) {
    prm.row_off[g] = pl.row_off[g];
    prm.tile_base[g] = pl.tile_base[g];
  }
  for (int g = 0; g < pl.num_groups; ++g)
    prm.group_alpha[g] = a.group_alpha ? a.group_alpha[g] : a.alpha;
#ifdef PETIT_CHECK_BOUNDS
  {
    const int64_t chunk = pl.fmt == kMXFP4 ? FmtTraits<kMXFP4>::kChunkBytes
                                           : FmtTraits<kNVFP4>::kChunkBytes;
    // (with CTA pairs a work tile holds two 128-row weight tiles)
    const int64_t wb = static_cast<int64_t>(pl.n_tiles) * (pl.pair ? 2 : 1) * pl.k_stages * chunk;
    const int64_t ce = static_cast<int64_t>(pl.row_off[pl.num_groups]) * a.n;
    const int64_t lw = g_check_weight_bytes.load(), lc = g_check_c_elems.load();
    prm.chk_rep_bytes = lw >= 0 && lw < wb ? lw : wb;
    prm.chk_c_elems = lc >= 0 && lc < ce ? lc : ce;
    prm.chk_a_rows = pl.row_off[pl.num_groups];
  }
#endif
  if (pl.fmt == kNVFP4)
    return launch_fmt<kNVFP4>(pl.bn, pl.ku, pl.pair, prm, tmap, stream, a.device);
  if (pl.fmt == kNVFP4F16)
    return launch_fmt<kNVFP4F16>(pl.bn, pl.ku, pl.pair, prm, tmap, stream, a.device);
  return launch_fmt<kMXFP4>(pl.bn, pl.ku, pl.pair, prm, tmap, stream, a.device);
}

}  // namespace petit
