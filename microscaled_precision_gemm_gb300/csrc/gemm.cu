// K2 / K3: block-scaled MXFP6 x MXFP6 GEMM on the 5th-generation tensor cores.
//
//   C[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k]        A: [M][K], B: [N][K], K-major
//
// "Optimizing Krea 3 on AMD Instinct MI355X", section "We built a faster MXFP6
// kernel" (Figure 1): the MLP's GEMMs run in MXFP6, with 6-bit values packed in
// memory (not one per byte) and no operand re-reads between neighbouring tiles.
// Section "Fusion cut intermediate memory traffic": the up-projection's epilogue
// writes the MXFP6 intermediate the down-projection reads directly.
//
// Design (sm_103a): a CTA pair (cluster of 2) computes a 256 x 256 output tile
// with the pair-wide MMA (tcgen05 cta_group::2). CTA r of the pair owns A rows
// [128 r, 128 r + 128) of the tile and B rows (output columns) [128 r, 128 r + 128);
// the tensor cores of both SMs read both halves of B, so each SM stages only half
// of B: 33.5 KB of shared memory per 128-deep K step, which leaves room for a
// 6-stage ring. Persistent: one pair per two SMs, walking tile pairs.
//   warp 0      TMA producer (each CTA): one 16U6 tiled load for its A rows, one
//               for its half of B (128-byte swizzle), and tiled loads of the scale
//               atoms its SM's tensor memory needs (its own A rows, all 256 B rows).
//               All four loads of both CTAs complete on the leader CTA's barrier,
//               which expects both CTAs' bytes (cta_group::2 TMA completion).
//   warp 1      leader CTA: once the stage's scales are in tensor memory (which
//               the scale warp signals only after the stage's operands landed),
//               issues four tcgen05.mma cta_group::2 kind::mxf8f6f4
//               block_scale per stage (M=256, N=256, K=32, E2M3 x E2M3, E8M0) into
//               each SM's fp32 accumulator (128 lanes x 256 columns).
//   warp 10     leader CTA: copies each stage's scale atoms into both SMs' tensor
//               memory (tcgen05.cp cta_group::2) in its own tcgen05 stream and
//               signals the MMA warp, so no MMA queues behind a copy.
//   warps 2-9   epilogue (each CTA): drain 32 rows x 128 columns of the local
//               accumulator into registers, release tensor memory to the leader at
//               once, then one of the fused epilogues:
//                 kEpiBf16      bias + BF16 store (the down-projection, K2)
//                 kEpiGelu      bias + tanh-GELU + MXFP6 requantization (K3)
//                 kEpiSwiglu    stacked gate/up weight: CTA 0 of the pair stages gate
//                               rows, CTA 1 the matching up rows, so accumulator
//                               columns c and 128 + c are gate and up of one output
//                               column; bias + silu(gate) * up + MXFP6 requantization
//                 kEpiGateRes   bias, times a per-column gate, plus a BF16 residual,
//                               BF16 store (an output projection with its gate and
//                               residual add)
//               Every epilogue stages its output in the warp's own 2 KB shared slot
//               and writes it with TMA tensor stores: a 32-row x 32-column BF16
//               block, or the 6-bit codes of two 32-column MX blocks (48 bytes) of
//               32 rows. Each thread storing its own row instead (a 16- or 8-byte
//               piece of 32 rows per store instruction) kept busy the
//               shared-memory pipe that the main loop's operand traffic needs.
//   warp 11     (QA instance only, each CTA) the in-kernel quantizer: encodes A's
//               BF16 rows to MXFP6 (the quantizer's rule and layout) while the
//               main loop runs, and publishes each 128-row block on a counter in
//               global memory; producers wait for a block's counter before their
//               first load of it (see QaArgs below).
// Every mbarrier wait suspends the waiting thread until its phase completes (a
// try_wait suspend-time hint: spinning waits took issue slots from the MMA and
// TMA threads) and is bounded (2 s on the global timer); on expiry the kernel
// records an error bit, drains its in-flight copies and MMAs (again bounded), frees
// tensor memory and returns. A second instance of the kernel (SPLIT) divides a
// nearly empty last round of tiles along K across all pairs (see Plan below);
// another (HALF) runs such a round's tiles as 128-column halves on twice the pairs
// (N = 128 pair MMAs), where the split tail is not taken. In the QA instance
// (warp 11 above) producers wait on other CTAs' quantizer warps, which claim their
// work from a counter, so only running CTAs hold any (see QaArgs below).
// Launched with programmatic dependent launch: the
// prologue (barriers, tensor memory, tensor-map prefetch) may overlap the previous
// kernel in the stream, and griddepcontrol.wait holds every access to global
// memory until that kernel has completed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "mx_layout.cuh"
#include "mx_quant.cuh"
#include "ptx.cuh"

namespace mxk {

__device__ unsigned int g_error_word;

enum : int { kEpiBf16 = 0, kEpiGelu = 1, kEpiSwiglu = 2, kEpiGateRes = 3 };

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int kStages = 6;
constexpr int kPair = 2;              // CTAs per cluster (one MMA pair)
constexpr uint16_t kPairMask = 0x3;
constexpr int kBHalfRows = BN / kPair;
constexpr int kEpiWarps = 8;                     // 2 per tensor-memory lane quadrant
constexpr int kEpiCols = BN * 4 / kEpiWarps;     // accumulator columns each epilogue warp drains
constexpr int kEpiChunks = kEpiCols / 32;        // 32-column MX blocks per epilogue thread
constexpr int kThreads = (3 + kEpiWarps) * 32;  // + scale-copy warp
constexpr int kQaWarp = 3 + kEpiWarps;           // the QA instance's quantizer warp
constexpr uint32_t kQaPauseNs = 1000;              // the quantizer warp's pause between groups
constexpr int kThreadsQa = kThreads + 32;
constexpr uint32_t kABytes = BM * BK;  // 16-byte shared slot per 16 codes -> 1 byte per element
constexpr uint32_t kBBytes = kBHalfRows * BK;   // this CTA's half of the B tile
constexpr uint32_t kSfaBytes = kAtomBytes;
constexpr uint32_t kSfbBytes = 2 * kAtomBytes;
// A 16U6 load writes the 12 data bytes of each 16-byte shared slot (the 4 padding
// bytes are left untouched), so it completes 3/4 of the slot bytes on the mbarrier.
constexpr uint32_t kStageTx = (kABytes + kBBytes) / 4 * 3 + kSfaBytes + kSfbBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = BN;  // scale slots after the accumulator: stage s at +16 s (A +0, B +8)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kOutBoxCols = 32;                                   // one epilogue chunk
constexpr uint32_t kOutStageBytes = 32 * kOutBoxCols * 2;         // 32 rows of BF16
constexpr uint32_t kCodesBoxBytes = 48;                           // two MX blocks of 6-bit codes
static_assert(32 * kCodesBoxBytes <= kOutStageBytes, "a codes box fits the store slot");

struct __align__(1024) SharedStorage {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint8_t sfa[kStages][kSfaBytes];
  uint8_t sfb[kStages][kSfbBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t sfready[kStages];   // leader: the stage's scales are in both SMs' tensor memory
  uint64_t tmem_full;
  uint64_t tmem_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float bias_s[kEpiWarps][kEpiCols];   // each epilogue warp's bias values (read as float4)
  alignas(16) float gate_s[kEpiWarps][kEpiCols];   // kEpiGateRes: each epilogue warp's gate values
  uint64_t res_full[kEpiWarps];   // kEpiGateRes: each epilogue warp's residual box has landed
  // each epilogue warp's output box (BF16 32 x 32 with a 64-byte swizzle, or 32
  // rows of 48 code bytes), the source of its TMA stores
  alignas(1024) uint8_t out_stage[kEpiWarps][kOutStageBytes];
};
constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024;
static_assert(offsetof(SharedStorage, bias_s) % 16 == 0 && offsetof(SharedStorage, gate_s) % 16 == 0,
              "bias and gate staging are read as float4");
static_assert(offsetof(SharedStorage, sfa) % 128 == 0 && offsetof(SharedStorage, sfb) % 128 == 0,
              "scale atoms are TMA destinations");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(offsetof(SharedStorage, out_stage) % 1024 == 0 && kOutStageBytes % 1024 == 0,
              "TMA store sources sit on 1024-byte boundaries (the 64-byte swizzle repeats every 512 bytes)");
static_assert(kPair * BM == kPairTileRows && BN == kPairTileCols && BK == kStepK, "tile geometry of the launch plan");
static_assert(kPair * kEpiWarps == kArrivalWordsPerTile, "one arrival counter per CTA and epilogue warp");
static_assert(kSplitSlotBytes == size_t{kPair} * kEpiWarps * kEpiChunks * 8 * 32 * sizeof(float4),
              "a partial slot holds both CTAs' accumulators");

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Descriptor of one 512-byte scale atom: 32 rows of 16 bytes, no swizzle,
// 8-row core matrices 128 B apart.
__device__ __forceinline__ uint64_t desc_scale_atom(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 32) |
         (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A, B = E2M3, K-major,
// fp32 accumulate, E8M0 scales, M = 256 (the pair), N = 256; j selects the scale byte
// (K-block) inside each 32-bit tensor-memory scale column, for A and B alike.
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t j, uint32_t n = BN) {
  return (j << 4) | (3u << 7) | (3u << 10) | ((n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>((kPair * BM) >> 4) << 24) | (j << 29);
}
constexpr int kHalfCols = BN / 2;   // a half tile's output columns
// A half tile's stage: all of this CTA's A rows, half of its B rows.
constexpr uint32_t kStageTxHalf = (kABytes + kBBytes / 2) / 4 * 3 + kSfaBytes + kSfbBytes;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned err_bit) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicOr(&g_error_word, err_bit);
        return false;
      }
    }
  }
}

// As wait_bounded, for barriers the peer CTA arrives on (acquire at cluster scope).
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                     unsigned err_bit) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicOr(&g_error_word, err_bit);
        return false;
      }
    }
  }
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      atomicOr(&g_error_word, kErrDrain);
      return;
    }
  }
}

// Work plan shared by every role. Tiles are pair tiles (256 rows x 256 columns,
// CTA r of the pair: row tile 2 p_m + r) in row-major order. Without a split
// tail, cluster c takes tiles c, c + #clusters, ... When the last round would
// leave most pairs idle (the host's rule: at most a quarter of a round left over,
// and long tiles), the first sk_tiles = #clusters + (tiles mod #clusters) tiles
// are shared out along K instead: their sk_tiles * kblocks K-steps are cut into
// one contiguous range per cluster (every cluster gets at least one tile's worth), and the
// remaining tiles, a whole number of rounds, are taken whole as above. A range
// boundary inside a tile makes it a split tile with exactly two contributors;
// each stores its fp32 partial accumulator, and whichever arrives second adds
// the other's partial and runs the epilogue. fp32 addition of two terms is
// commutative, so the result does not depend on which one that is.
struct Plan {
  int tiles, num_n, kblocks, clusters, sk_tiles;
  int whole;        // tiles run whole (tiles - half_tiles)
  int half_tiles;   // trailing tiles run as two halves: half unit c < 2 half_tiles of cluster c
  float4* partial;     // split tiles: 2 slots per cluster, each 2 CTAs x 128 rows x 256 fp32
  unsigned* arrivals;  // split tiles: arrivals per (tile, CTA rank, epilogue warp); zero before the launch
};

// A stretch of one tile's K-steps [kb0, kb1) that one cluster computes.
struct Unit {
  int tile, kb0, kb1;
};

// A cluster's split range, in K-steps counted from the start of tile 0 (the host
// keeps sk_tiles * kblocks below 2^31).
struct Cursor {
  int pos, end;
};

// First K-step of cluster c's split range.
__device__ __forceinline__ int split_start(const Plan& pl, int c) {
  return static_cast<int>(static_cast<int64_t>(pl.sk_tiles) * pl.kblocks * c / pl.clusters);
}

__device__ __forceinline__ Cursor cursor_begin(const Plan& pl, int c) {
  Cursor k;
  k.pos = split_start(pl, c);
  k.end = split_start(pl, c + 1);
  return k;
}

// The next unit of the split range. Every role walks the same sequence: the
// split range first (so the exchange of partials overlaps the whole tiles that
// follow), then whole tiles sk_tiles + c, sk_tiles + c + #clusters, ... in a loop
// of their own, which carries none of the split state.
__device__ __forceinline__ bool cursor_next(const Plan& pl, Cursor& k, Unit& u) {
  if (k.pos < k.end) {
    const int t = k.pos / pl.kblocks;
    const int lo = t * pl.kblocks;
    u.tile = t;
    u.kb0 = k.pos - lo;
    u.kb1 = min(k.end - lo, pl.kblocks);
    k.pos = lo + u.kb1;
    return true;
  }
  return false;
}

// In-kernel quantizer (QA instance). The rows of row blocks [0, first_block) were
// encoded before the launch; the rest -- rows up to M rounded up to 128, padding
// rows getting zero scales -- are cut into items of one row's 1024-column strip
// (one 32-element block per lane, as the quantize kernel encodes them), groups of
// kQaGroup items in row order. The quantizer warps claim groups in turn from a
// work counter (an atomic add on counter word 0: block 0 lies in the leading rows,
// first_block >= 2, so no producer reads it). Each group is published on its
// 128-row block's counter (release after the stores); a producer acquires the
// counter of its A row block, until it reads 128 x strips, before the first TMA
// load of that block. The counters are zero at the launch (the quantize kernel
// before it zeroes them). A quantizer warp waits on nothing and claims groups until
// none is left, so every claimed group is published whatever the other roles do,
// and a group is claimed only by a CTA that is running: no producer waits on a CTA
// that has not started, and the launch needs no co-residency guarantee.
struct QaArgs {
  const uint16_t* x;   // BF16 A [M][K], row stride ld_x elements
  int64_t ld_x;
  uint8_t* codes;      // the A operand the tensor maps read
  uint8_t* scales;
  unsigned* ready;     // one counter per 128-row block
  int first_block;
  int strips;          // 1024-column strips per row
  int wide;            // x and its row stride 32-byte aligned: 32-byte loads
};

// Producer side: acquire the counter of A row block mb until it reads 128 x strips
// (every item of the block published), then a proxy fence so that the tensor loads
// that follow read the block. False when the wait gave up.
__device__ __forceinline__ bool acquire_quantized(const QaArgs& qa, int mb, volatile int* abort_flag) {
  const uint32_t target = 128u * static_cast<uint32_t>(qa.strips);
  const unsigned* c = qa.ready + mb;
  if (ld_acquire_gpu(c) < target) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; ld_acquire_gpu(c) < target; ++i) {
      sleep_ns(200);
      if ((i & 15) == 0) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
          *abort_flag = 1;
          atomicOr(&g_error_word, kErrWaitQuant);
          return false;
        }
      }
    }
  }
  fence_proxy_async_global();
  return true;
}

// The quantizer warp (all 32 lanes). An item is one row's 1024-column strip (2 KB
// of BF16); lane l encodes its K-block 32 s + l (64 contiguous bytes) with the
// quantize kernel's block encoder. Memory instructions per item are kept few
// (they share the SM's memory pipeline with the main loop): two 32-byte loads per
// lane where x allows them (wide: 32-byte aligned rows), else four 16-byte loads;
// the lane's 24 code bytes as one 16-byte and one 8-byte store (which comes first
// depends on the lane's 8-byte phase); one 4-byte scale word per four lanes. Loads
// of a group's kQaGroup items are issued together.
__device__ __forceinline__ void run_quantizer(const QaArgs& qa, int m_total, int k_total, int lane) {
  const uint32_t strips = static_cast<uint32_t>(qa.strips);
  const uint32_t kblocks = static_cast<uint32_t>(k_total / kBlock);
  const uint32_t first = static_cast<uint32_t>(qa.first_block) * 128u * strips;
  const uint32_t items = static_cast<uint32_t>(pad_rows(m_total)) * strips;
  const uint32_t groups = items > first ? (items - first) / kQaGroup : 0u;
  const int64_t pitch = static_cast<int64_t>(k_total) / 4 * 3;
  const bool odd = (lane & 1) != 0;   // the lane's codes start 8 bytes into a 16-byte unit
  // the next group is claimed while the current one is encoded (a warp claims one
  // past the end before it stops)
  unsigned claim = lane == 0 ? atomicAdd(qa.ready, 1u) : 0u;
  for (uint32_t q = __shfl_sync(0xffffffffu, claim, 0); q < groups; q = __shfl_sync(0xffffffffu, claim, 0)) {
    claim = lane == 0 ? atomicAdd(qa.ready, 1u) : 0u;
    const uint32_t i0 = first + q * kQaGroup;
    uint4 raw[kQaGroup][4];
    uint32_t row[kQaGroup], kb[kQaGroup];
#pragma unroll
    for (int g = 0; g < kQaGroup; ++g) {
      row[g] = (i0 + g) / strips;
      kb[g] = ((i0 + g) - row[g] * strips) * 32u + lane;
      const bool live = row[g] < static_cast<uint32_t>(m_total) && kb[g] < kblocks;
      const uint16_t* src = qa.x + static_cast<int64_t>(row[g]) * qa.ld_x + kb[g] * 32u;
      if (!live) {
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[g][j] = make_uint4(0, 0, 0, 0);
      } else if (qa.wide) {
        ld_nc_v8(src, raw[g][0], raw[g][1]);
        ld_nc_v8(src + 16, raw[g][2], raw[g][3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[g][j] = ld_nc(src + 8 * j);
      }
    }
#pragma unroll
    for (int g = 0; g < kQaGroup; ++g) {
      // BF16 -> fp32 is exact, so the fp32 block encoder gives the BF16 rule's result;
      // a padding row's zeros give a zero scale
      float f[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v[4] = {raw[g][j].x, raw[g][j].y, raw[g][j].z, raw[g][j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f[8 * j + 2 * i] = __uint_as_float(v[i] << 16);
          f[8 * j + 2 * i + 1] = __uint_as_float(v[i] & 0xFFFF0000u);
        }
      }
      uint32_t w[6];
      const uint32_t sc = quant_block32(f, w);
      // four consecutive lanes (K-blocks 4c .. 4c + 3 of the row) -> one tiled scale word;
      // the strip's valid lanes come in whole fours (K % 128 == 0)
      const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 1);
      const uint32_t s2 = __shfl_down_sync(0xffffffffu, sc, 2);
      const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 3);
      if (kb[g] < kblocks) {
        if ((lane & 3) == 0)
          *reinterpret_cast<uint32_t*>(qa.scales + scale_word_offset(row[g], kb[g] / 4, k_total)) =
              sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
        if (row[g] < static_cast<uint32_t>(m_total)) {
          // 24 bytes at 24 kb: 16-byte aligned for an even lane (16 + 8 bytes), 8 bytes
          // past a 16-byte boundary for an odd one (8 + 16 bytes)
          uint8_t* d = qa.codes + static_cast<int64_t>(row[g]) * pitch + kb[g] * 24u;
          *reinterpret_cast<uint4*>(d + (odd ? 8 : 0)) =
              odd ? make_uint4(w[2], w[3], w[4], w[5]) : make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint2*>(d + (odd ? 0 : 16)) = odd ? make_uint2(w[0], w[1]) : make_uint2(w[4], w[5]);
        }
      }
    }
    // the group's four items lie in one 128-row block (128 x strips is a multiple of 4)
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0) red_release_gpu_add(qa.ready + i0 / strips / 128u, kQaGroup);
    // a pause between groups spreads the warp's memory instructions over more of the
    // main loop, which shares the SM's memory pipeline with them: 1 us took 1 and 2.7
    // us off the M = 4096 and 20480 up-projections; 1.5 us and more fell behind the
    // GEMM's reads (measured)
    sleep_ns(kQaPauseNs);
  }
}

__device__ __forceinline__ void pair_tile(const Plan& pl, int tile, int rank, int* mb, int* nb) {
  const int pm = tile / pl.num_n;
  *nb = tile - pm * pl.num_n;
  *mb = pm * kPair + rank;
}

// gated: B is the stacked [gate; up] weight of 2 * n_out rows; CTA 0 of the pair
// stages gate rows [128 nb, 128 nb + 128) and CTA 1 the up rows n_out rows further,
// and both SMs' tensor memory gets the scale atoms of both row groups.
// HALF: half units (the cluster's after its whole tiles) load half of this CTA's B
// rows through tbh (64-row boxes) and the one scale atom of the half's 128 rows.
template <bool SPLIT, bool QA, bool HALF>
__device__ __forceinline__ void run_producer(SharedStorage& s, const CUtensorMap* ta, const CUtensorMap* tb,
                                             const CUtensorMap* tbh, const CUtensorMap* tsa, const CUtensorMap* tsb,
                                             const Plan& pl, int cluster, int rank, bool gated, int n_out,
                                             const QaArgs& qa, int num_m, volatile int* abort_flag) {
  const int kblocks = pl.kblocks;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t filled = 0, fill_parity = 0;
  bool ok = true;
  // QA: the A row block acquired last. A tile's block is acquired right before the
  // tile's first load (measured: an acquire read issued a tile ahead, after the
  // first load, drained the ring; batched relaxed reads with one acquire fence cost
  // more than this read). Blocks below first_block were encoded before the launch;
  // a block past M has no rows.
  int acquired_mb = -1;
  auto quantized = [&](int mb) { return mb < qa.first_block || mb >= num_m || mb == acquired_mb; };
  auto load_unit = [&](int tile, int kb0, int kb1, int half) {
    const bool is_half = HALF && half >= 0;
    int mb, nb;
    pair_tile(pl, tile, rank, &mb, &nb);
    if constexpr (QA) {
      if (!quantized(mb)) {
        if (!acquire_quantized(qa, mb, abort_flag)) {
          ok = false;
          return;
        }
        acquired_mb = mb;
      }
    }
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!wait_bounded(&s.empty[stage], phase ^ 1u, abort_flag, kErrWaitProducer)) {
        ok = false;
        return;
      }
      // both CTAs' stage bytes complete on the leader's full barrier, which
      // expects them all; a row tile past M reads zeros (A and its scales)
      const uint32_t full_leader = mapa_shared(smem_u32(&s.full[stage]), 0);
      if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], kPair * (is_half ? kStageTxHalf : kStageTx));
      tma_load_2d_pair(s.a[stage], ta, full_leader, kb * BK, mb * BM);
      if (is_half) {
        // CTA r: rows [64 r, 64 r + 64) of the half's 128 B rows; the second atom of
        // the two-atom scale box is the next half's (zeros past N), unused
        tma_load_2d_pair(s.b[stage], tbh, full_leader, kb * BK, nb * BN + half * kHalfCols + rank * (kHalfCols / 2));
        tma_load_2d_pair(s.sfa[stage], tsa, full_leader, 0, mb * kblocks + kb);
        tma_load_3d_pair(s.sfb[stage], tsb, full_leader, 0, kb, 2 * nb + half);
      } else {
      const int b_row = gated ? rank * n_out + nb * kBHalfRows : nb * BN + rank * kBHalfRows;
      tma_load_2d_pair(s.b[stage], tb, full_leader, kb * BK, b_row);
      tma_load_2d_pair(s.sfa[stage], tsa, full_leader, 0, mb * kblocks + kb);
      if (gated) {
        tma_load_3d_pair(s.sfb[stage], tsb, full_leader, 0, kb, nb);
        tma_load_3d_pair(s.sfb[stage] + kAtomBytes, tsb, full_leader, 0, kb, n_out / kBHalfRows + nb);
      } else {
        tma_load_3d_pair(s.sfb[stage], tsb, full_leader, 0, kb, 2 * nb);
      }
      }
      filled |= 1u << stage;
      fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  };
  if constexpr (SPLIT) {
    Cursor cur = cursor_begin(pl, cluster);
    Unit u;
    while (ok && cursor_next(pl, cur, u)) load_unit(u.tile, u.kb0, u.kb1, -1);
  }
  for (int p = (SPLIT ? pl.sk_tiles : 0) + cluster; ok && p < (HALF ? pl.whole : pl.tiles); p += pl.clusters)
    load_unit(p, 0, kblocks, -1);
  if constexpr (HALF) {
    if (ok && cluster < 2 * pl.half_tiles) load_unit(pl.whole + cluster / 2, 0, kblocks, cluster % 2);
  }
  if (ok) {
    // every stage this CTA filled has been consumed by the pair's MMAs, so no
    // completion arrival from the leader is still heading here
    for (int st = 0; st < kStages; ++st)
      if ((filled >> st) & 1u) wait_drain(&s.empty[st], (fill_parity >> st) & 1u);
  } else if (rank == 0) {
    for (int st = 0; st < kStages; ++st)
      if ((filled >> st) & 1u) wait_drain(&s.full[st], (fill_parity >> st) & 1u);
  }
}

// HALF: a half unit's MMAs are N = 128 (accumulator columns 0-127; the B scales
// of its 128 rows are the first atom of the stage's scale slot).
template <bool SPLIT, bool HALF>
__device__ __forceinline__ void run_mma(SharedStorage& s, uint32_t tmem, const Plan& pl, int cluster,
                                        volatile int* abort_flag) {
  int stage = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool ok = true, issued = false;
  auto mma_unit = [&](int kb0, int kb1, bool half) {
    const uint32_t n = HALF && half ? static_cast<uint32_t>(kHalfCols) : static_cast<uint32_t>(BN);
    // both CTAs' epilogues have drained the previous tile's accumulators
    if (!wait_bounded_cluster(&s.tmem_empty, acc_phase ^ 1u, abort_flag, kErrWaitMma)) {
      ok = false;
      return;
    }
    tc_fence_after();
    for (int kb = kb0; kb < kb1; ++kb) {
      // scales copied into both SMs' tensor memory, and therefore operands landed:
      // the scale warp copies a stage only after its own wait on full[stage] (which
      // both CTAs' operand loads complete), and its commit arrives on sfready after
      // those copies, so acquiring sfready orders this thread after the operand
      // writes too. One wait per K-step instead of two (measured ~1% faster).
      if (!wait_bounded(&s.sfready[stage], phase, abort_flag, kErrWaitMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const uint32_t sf_a = tmem + kSfCol0 + 16u * stage;
        const uint32_t sf_b = sf_a + 8u;
        const uint64_t ad = desc_sw128(smem_u32(s.a[stage]));
        const uint64_t bd = desc_sw128(smem_u32(s.b[stage]));
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j) {
          // K step j: 32 elements = 32 bytes further along the swizzled 128-byte row
          tc_mma_mx_pair(tmem, ad + 2u * j, bd + 2u * j, idesc_mx(j, n), sf_a, sf_b, (kb != kb0) || j != 0);
        }
        tc_commit_pair(&s.empty[stage], kPairMask);  // frees the stage in both CTAs
        issued = true;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) return;
    tc_commit_pair(&s.tmem_full, kPairMask);
    acc_phase ^= 1u;
  };
  if constexpr (SPLIT) {
    Cursor cur = cursor_begin(pl, cluster);
    Unit u;
    while (ok && cursor_next(pl, cur, u)) mma_unit(u.kb0, u.kb1, false);
  }
  for (int p = (SPLIT ? pl.sk_tiles : 0) + cluster; ok && p < (HALF ? pl.whole : pl.tiles); p += pl.clusters)
    mma_unit(0, pl.kblocks, false);
  if constexpr (HALF) {
    if (ok && cluster < 2 * pl.half_tiles) mma_unit(0, pl.kblocks, true);
  }
  if (!ok && issued) {
    tc_commit_pair(&s.drain, 0x1);
    wait_drain(&s.drain, 0);
  }
}

// Leader CTA, scale warp: copies each stage's scale atoms into both SMs' tensor
// memory in its own tcgen05 stream and signals sfready[stage] when they landed.
template <bool SPLIT, bool HALF>
__device__ __forceinline__ void run_scales(SharedStorage& s, uint32_t tmem, const Plan& pl, int cluster,
                                           volatile int* abort_flag) {
  // the split range's K-steps, then kblocks per whole tile, then per half unit
  const int first_whole = (SPLIT ? pl.sk_tiles : 0) + cluster;
  const int end = HALF ? pl.whole : pl.tiles;
  const int64_t whole = first_whole < end ? (end - first_whole + pl.clusters - 1) / pl.clusters : 0;
  int64_t steps = whole * pl.kblocks;
  if constexpr (SPLIT) steps += split_start(pl, cluster + 1) - split_start(pl, cluster);
  if constexpr (HALF) steps += cluster < 2 * pl.half_tiles ? pl.kblocks : 0;
  int stage = 0;
  uint32_t phase = 0;
  for (int64_t g = 0; g < steps; ++g) {
    if (!wait_bounded(&s.full[stage], phase, abort_flag, kErrWaitMma)) return;
    tc_fence_after();
    const uint32_t sf_a = tmem + kSfCol0 + 16u * stage;
    const uint32_t sf_b = sf_a + 8u;
    tc_cp_pair_32x128b_warpx4(sf_a, desc_scale_atom(smem_u32(s.sfa[stage])));
    tc_cp_pair_32x128b_warpx4(sf_b, desc_scale_atom(smem_u32(s.sfb[stage])));
    tc_cp_pair_32x128b_warpx4(sf_b + 4u, desc_scale_atom(smem_u32(s.sfb[stage] + kAtomBytes)));
    tc_commit_pair(&s.sfready[stage], 0x1);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

// One epilogue warp stages kEpiCols fp32 values of a BF16 vector in shared memory:
// lanes 0-15 convert 4 consecutive values each from src[n_lo ...], lanes 16-31 from
// src[n_hi ...] (n_hi = n_lo + 64 for a contiguous range); a null src stages `fill`.
// Chunks then read them as broadcasts.
__device__ __forceinline__ void stage_vec(float* bw, const uint16_t* __restrict__ src, int n_lo, int n_hi, int lane,
                                          float fill) {
  static_assert(kEpiCols == 128, "two halves of 64 values, 4 per lane");
  float f[4] = {fill, fill, fill, fill};
  if (src != nullptr) {
    const int n = (lane < 16 ? n_lo : n_hi) + 4 * (lane & 15);
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src + n));
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
  __syncwarp();  // the previous tile's reads are done
  *reinterpret_cast<float4*>(bw + 4 * lane) = make_float4(f[0], f[1], f[2], f[3]);
  __syncwarp();
}

// Values 4 v .. 4 v + 3 of staged chunk c (32 values per chunk).
__device__ __forceinline__ float4 staged4(const float* bw, int c, int v) {
  return reinterpret_cast<const float4*>(bw + 32 * c)[v];
}

// With u = sqrt(2/pi) (v + 0.044715 v^3), exp(-2u) = 2^t for
// t = v (kGeluC2 + kGeluC1 v^2): kGeluC2 = -2 sqrt(2/pi) log2(e), kGeluC1 = 0.044715 kGeluC2.
// For very negative v, 2^t is +inf and the result is v * 0 = -0 (the exact value
// there is below 1e-37 in magnitude).
constexpr float kGeluC2 = -2.0f * 0.7978845608028654f * 1.4426950408889634f;
constexpr float kGeluC1 = 0.044715f * kGeluC2;

__device__ __forceinline__ float gelu_tanh(float v) {
  const float t = v * fmaf(kGeluC1, v * v, kGeluC2);
  return v * rcp_approx(1.0f + ex2_approx(t));
}

// gelu_tanh of a packed pair, rounding exactly as the scalar form: the multiplies,
// the fma and the add run two-wide, 2^t and the reciprocal per lane.
__device__ __forceinline__ void gelu_tanh2(uint64_t v, float& g0, float& g1) {
  const uint64_t t = f2_mul(v, f2_fma(f2_mul(v, v), f2_pack(kGeluC1, kGeluC1), f2_pack(kGeluC2, kGeluC2)));
  float t0, t1;
  f2_unpack(t, t0, t1);
  float d0, d1;
  f2_unpack(f2_add(f2_pack(ex2_approx(t0), ex2_approx(t1)), f2_pack(1.0f, 1.0f)), d0, d1);
  f2_unpack(f2_mul(v, f2_pack(rcp_approx(d0), rcp_approx(d1))), g0, g1);
}

// silu(v) = v / (1 + e^-v) = v / (1 + 2^(-v log2 e)). For very negative v, 2^.. is
// +inf and the result is v * 0 = -0 (the exact value is below 1e-37 in magnitude).
constexpr float kNegLog2e = -1.4426950408889634f;

__device__ __forceinline__ float silu(float v) { return v * rcp_approx(1.0f + ex2_approx(v * kNegLog2e)); }

// silu(g) * u of packed pairs, rounding exactly as the scalar form.
__device__ __forceinline__ void silu_mul2(uint64_t g, uint64_t u, float& h0, float& h1) {
  float t0, t1;
  f2_unpack(f2_mul(g, f2_pack(kNegLog2e, kNegLog2e)), t0, t1);
  float d0, d1;
  f2_unpack(f2_add(f2_pack(ex2_approx(t0), ex2_approx(t1)), f2_pack(1.0f, 1.0f)), d0, d1);
  f2_unpack(f2_mul(f2_mul(g, f2_pack(rcp_approx(d0), rcp_approx(d1))), u), h0, h1);
}

__device__ __forceinline__ void store_dbg32(float* d, const float (&g)[32]) {
  float4* p = reinterpret_cast<float4*>(d);
#pragma unroll
  for (int v = 0; v < 8; ++v) p[v] = make_float4(g[4 * v], g[4 * v + 1], g[4 * v + 2], g[4 * v + 3]);
}

// Accumulator column (inside the 256-column tile) of epilogue chunk c of column group h.
// kEpiSwiglu: chunks 0, 1 are gate columns 64 h + 32 c, chunks 2, 3 the up columns 128 further.
template <int EPI>
__device__ __forceinline__ uint32_t chunk_col(int h, int c) {
  if constexpr (EPI == kEpiSwiglu)
    return static_cast<uint32_t>((c >> 1) * kBHalfRows + 64 * h + 32 * (c & 1));
  else
    return static_cast<uint32_t>(h * kEpiCols + 32 * c);
}

// A split tile: this warp stores its 32 rows x 128 columns of the partial
// accumulator, counts its arrival, and if the other contributor's part is
// already stored, adds it. Returns true when r holds the tile's full sum (this
// warp arrived second), false when the other contributor will finish the tile.
// Each epilogue warp has its own arrival counter, so no warp ever waits for another.
__device__ __forceinline__ bool split_exchange(const Plan& pl, int cluster, int rank, int ew, int lane,
                                               const Unit& u, uint32_t (&r)[kEpiChunks][32]) {
  const int lo = u.tile * pl.kblocks;
  const int64_t w = static_cast<int64_t>(pl.sk_tiles) * pl.kblocks;
  // the two contributors: the cluster whose range holds the tile's first K-step, and the next one
  const int first = static_cast<int>((static_cast<int64_t>(lo + 1) * pl.clusters - 1) / w);
  const int other = cluster == first ? first + 1 : first;
  // two slots per cluster: the tile its range starts in (0) and the tile it ends in (1)
  const int mine_slot = 2 * cluster + (split_start(pl, cluster) >= lo ? 0 : 1);
  const int other_slot = 2 * other + (split_start(pl, other) >= lo ? 0 : 1);
  constexpr int kVec = kEpiChunks * 8;  // float4 values per thread
  constexpr int64_t kSlot = static_cast<int64_t>(kPair) * kEpiWarps * kVec * 32;
  const int64_t base = (static_cast<int64_t>(rank) * kEpiWarps + ew) * kVec * 32 + lane;
  float4* mine = pl.partial + mine_slot * kSlot + base;
#pragma unroll
  for (int c = 0; c < kEpiChunks; ++c)
#pragma unroll
    for (int v = 0; v < 8; ++v)
      __stcg(mine + (c * 8 + v) * 32, make_float4(__uint_as_float(r[c][4 * v]), __uint_as_float(r[c][4 * v + 1]),
                                                  __uint_as_float(r[c][4 * v + 2]),
                                                  __uint_as_float(r[c][4 * v + 3])));
  __threadfence();
  __syncwarp();
  unsigned* counter = pl.arrivals + (static_cast<int64_t>(u.tile) * kPair + rank) * kEpiWarps + ew;
  unsigned old = 0;
  if (lane == 0) old = atomicAdd(counter, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == 0) return false;
  __threadfence();
  const float4* theirs = pl.partial + other_slot * kSlot + base;
#pragma unroll
  for (int c = 0; c < kEpiChunks; ++c)
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 o = __ldcg(theirs + (c * 8 + v) * 32);
      r[c][4 * v] = __float_as_uint(__uint_as_float(r[c][4 * v]) + o.x);
      r[c][4 * v + 1] = __float_as_uint(__uint_as_float(r[c][4 * v + 1]) + o.y);
      r[c][4 * v + 2] = __float_as_uint(__uint_as_float(r[c][4 * v + 2]) + o.z);
      r[c][4 * v + 3] = __float_as_uint(__uint_as_float(r[c][4 * v + 3]) + o.w);
    }
  if (lane == 0) *counter = 0u;  // both arrivals are in: zero again for the next launch
  return true;
}

// Epilogue state of one warp that stays the same from tile to tile.
struct EpiCtx {
  int warp, lane, q, h, rank, cluster;
  int num_m, m_total, n_total, n_out;
  uint32_t tmem, tmem_empty_leader;
  float* bw;
  float* gw;
  const CUtensorMap* tmap_out;   // the output: BF16 boxes of 32 x 32 (64-byte swizzle) or
                                 // 6-bit codes in boxes of 32 rows x 48 bytes
  const CUtensorMap* tmap_res;   // kEpiGateRes: the residual, boxes as the BF16 output's
  uint8_t* ostage;               // this warp's TMA store source (and residual box)
  uint64_t* res_bar;             // kEpiGateRes: completes when the residual box has landed
  uint32_t res_phase;            // its next phase parity
};

// The epilogue of one output tile (or, SPLIT, of one unit of the split region):
// drain the accumulator, release it, then the fused epilogue. Returns false when
// a wait gave up. n_total: the GEMM's N (rows of B; stacked 2 F for kEpiSwiglu);
// output width F = n_total / 2 for kEpiSwiglu, else n_total.
// col_tile: the unit's first output column (nb * BN for a whole tile; a half tile's
// 128 columns are drained by the warps of column group 0).
template <int EPI, bool DBG, bool SPLIT>
__device__ __forceinline__ bool epilogue_tile(SharedStorage& s, EpiCtx& e, int mb, int nb, int col_tile,
                                              uint32_t& acc_phase,
                                              const Plan& pl, const Unit& u, const uint16_t* __restrict__ bias,
                                              const uint16_t* __restrict__ gate, const uint16_t* residual, void* out,
                                              uint8_t* __restrict__ out_scales, float* __restrict__ dbg,
                                              volatile int* abort_flag) {
  const int lane = e.lane, q = e.q, h = e.h, warp = e.warp, rank = e.rank, cluster = e.cluster;
  const int num_m = e.num_m, m_total = e.m_total, n_total = e.n_total, n_out = e.n_out;
  const uint32_t tmem = e.tmem, tmem_empty_leader = e.tmem_empty_leader;
  float* bw = e.bw;
  float* gw = e.gw;
  // first output column of this warp: 64 of them (kEpiSwiglu) or 128
  const int col0 = (EPI == kEpiSwiglu) ? nb * kBHalfRows + 64 * h : col_tile + h * kEpiCols;
  if constexpr (EPI == kEpiSwiglu)
    stage_vec(bw, bias, col0, n_out + col0, lane, 0.f);
  else
    stage_vec(bw, bias, col0, col0 + 64, lane, 0.f);
  if constexpr (EPI == kEpiGateRes) {
    stage_vec(gw, gate, col0, col0 + 64, lane, 1.f);
    // the residual boxes this warp loads after the drain: its row's 128 columns into
    // L2 now, while the tile's main loop runs
    const int64_t prow = static_cast<int64_t>(mb) * BM + 32 * q + lane;
    if (prow < m_total) prefetch_l2_bulk(residual + prow * n_total + col0, kEpiCols * 2);
  }
  // kEpiGateRes: the first residual box is loaded while the warp waits for the
  // accumulator (once the previous tile's last store has read the slot)
  const bool box_live = static_cast<int64_t>(mb) * BM + 32 * q < m_total;
  bool res_pending = false;
  if constexpr (EPI == kEpiGateRes) {
    if (box_live) {
      if (lane == 0) {
        bulk_wait_read_all();
        mbar_arrive_expect_tx(e.res_bar, kOutStageBytes);
        tma_load_2d(e.ostage, e.tmap_res, e.res_bar, col0, static_cast<int32_t>(static_cast<int64_t>(mb) * BM + 32 * q));
      }
      res_pending = true;
    }
  }
  int ok = 0;
  if (lane == 0) ok = wait_bounded(&s.tmem_full, acc_phase, abort_flag, kErrWaitEpilogue) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) {
    if (res_pending && lane == 0) wait_drain(e.res_bar, e.res_phase);   // not in flight when the CTA leaves
    return false;
  }
  tc_fence_after();
  uint32_t r[kEpiChunks][32];
  const uint32_t t0 = tmem + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll
  for (int c = 0; c < kEpiChunks; ++c) tc_ld_32x32b_x32(t0 + chunk_col<EPI>(h, c), r[c]);
  tc_wait_ld();
  tc_fence_before();
  __syncwarp();
  // tcgen05.wait::ld has completed this warp's reads and the fence above orders
  // them before the signal; no memory is handed over, so the arrive is relaxed
  // (a release would first wait for the previous tile's global stores).
  if (lane == 0) mbar_arrive_remote_relaxed(tmem_empty_leader);
  acc_phase ^= 1u;
  if constexpr (SPLIT) {
    // a split tile's first contributor only stores its partial sum
    if ((u.kb0 != 0 || u.kb1 != pl.kblocks) && !split_exchange(pl, cluster, rank, warp - 2, lane, u, r)) {
      if (res_pending) {   // the first residual box is not used: let it land
        if (lane == 0) wait_drain(e.res_bar, e.res_phase);
        e.res_phase ^= 1u;
      }
      return true;
    }
  }

  const int64_t row0 = static_cast<int64_t>(mb) * BM + 32 * q;   // the warp's first row
  const int64_t row = row0 + lane;
  const bool live = row < m_total;
  if constexpr (EPI == kEpiBf16 || EPI == kEpiGateRes) {
#pragma unroll
    for (int c = 0; c < kEpiChunks; ++c) {
      const int n = col0 + 32 * c;
      uint32_t rw[16];  // kEpiGateRes: the residual's 32 BF16 values, two per word
      // 16-byte piece j of row `lane` sits at piece j ^ ((lane >> 1) & 3) of the row in
      // the warp's box (the 64-byte swizzle of the TMA boxes)
      uint4* srow = reinterpret_cast<uint4*>(e.ostage + lane * (kOutBoxCols * 2));
      if constexpr (EPI == kEpiGateRes) {
        // The residual box (these 32 rows x 32 columns) arrives by TMA in the warp's
        // store slot, once the previous store has read it, and is read back by rows:
        // per-row 16-byte global loads would touch 32 lines per warp instruction in
        // the SM's data pipe, which the main loop's operand traffic shares. The
        // output may be this very residual (in place): the box is read before the
        // same warp stores it.
        if (c > 0 && lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 16; ++j) rw[j] = 0u;
        if (box_live) {
          int got = 0;
          if (lane == 0) {
            if (c > 0) {   // chunk 0's box was loaded before the drain
              mbar_arrive_expect_tx(e.res_bar, kOutStageBytes);
              tma_load_2d(e.ostage, e.tmap_res, e.res_bar, n, static_cast<int32_t>(row0));
            }
            got = wait_bounded(e.res_bar, e.res_phase, abort_flag, kErrWaitEpilogue) ? 1 : 0;
            if (!got) wait_drain(e.res_bar, e.res_phase);   // the box is not in flight when the CTA leaves
          }
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) return false;
          // every lane observes the completed phase (lane 0 has seen it complete, and it
          // cannot advance before lane 0 arms it again) before reading the box
          for (int i = 0; i < 64 && !mbar_try_wait(smem_u32(e.res_bar), e.res_phase); ++i) {
          }
          e.res_phase ^= 1u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 v = srow[j ^ ((lane >> 1) & 3)];
            rw[4 * j] = v.x;
            rw[4 * j + 1] = v.y;
            rw[4 * j + 2] = v.z;
            rw[4 * j + 3] = v.w;
          }
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 b4 = staged4(bw, c, v);
        uint64_t x01 = f2_add(f2_pack(__uint_as_float(r[c][4 * v]), __uint_as_float(r[c][4 * v + 1])),
                              f2_pack(b4.x, b4.y));
        uint64_t x23 = f2_add(f2_pack(__uint_as_float(r[c][4 * v + 2]), __uint_as_float(r[c][4 * v + 3])),
                              f2_pack(b4.z, b4.w));
        if constexpr (EPI == kEpiGateRes) {
          const float4 g4 = staged4(gw, c, v);
          x01 = f2_fma(f2_pack(g4.x, g4.y), x01,
                       f2_pack(__uint_as_float(rw[2 * v] << 16), __uint_as_float(rw[2 * v] & 0xFFFF0000u)));
          x23 = f2_fma(f2_pack(g4.z, g4.w), x23,
                       f2_pack(__uint_as_float(rw[2 * v + 1] << 16), __uint_as_float(rw[2 * v + 1] & 0xFFFF0000u)));
        }
        float x0, x1, x2, x3;
        f2_unpack(x01, x0, x1);
        f2_unpack(x23, x2, x3);
        pk[2 * v] = cvt_bf16x2(x1, x0);
        pk[2 * v + 1] = cvt_bf16x2(x3, x2);
      }
      if constexpr (EPI != kEpiGateRes) {
        // the slot is free once the warp's previous store has read it
        if (lane == 0) bulk_wait_read_all();
      }
      // (kEpiGateRes: every lane has read its row of the residual box)
      __syncwarp();
      // the swizzle puts the warp's 16-byte writes on distinct banks
#pragma unroll
      for (int j = 0; j < 4; ++j)
        srow[j ^ ((lane >> 1) & 3)] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      // rows past M in the box are not written; a box wholly past M is not issued
      if (lane == 0 && row0 < m_total) {
        tma_store_2d(e.tmap_out, e.ostage, n, static_cast<int32_t>(row0));
        bulk_commit_group();
      }
    }
  } else {
    // MXFP6 requantization along the output columns, one 32-column block at a time
    constexpr int kBlocks = (EPI == kEpiSwiglu) ? kEpiChunks / 2 : kEpiChunks;
    static_assert(kBlocks % 2 == 0, "codes leave in boxes of two 32-column blocks");
    uint32_t scale_word = 0;
    uint32_t wprev[6];   // the codes of the first block of each pair
#pragma unroll
    for (int c = 0; c < kBlocks; ++c) {
      const int n = col0 + 32 * c;
      float g[32];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 b4 = staged4(bw, c, v);
        const uint64_t bb[2] = {f2_pack(b4.x, b4.y), f2_pack(b4.z, b4.w)};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = 4 * v + 2 * t;
          const uint64_t x = f2_add(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), bb[t]);
          if constexpr (EPI == kEpiGelu) {
            gelu_tanh2(x, g[i], g[i + 1]);
          } else {
            const float4 u4 = staged4(bw, 2 + c, v);
            const uint64_t bu = t == 0 ? f2_pack(u4.x, u4.y) : f2_pack(u4.z, u4.w);
            const uint64_t u = f2_add(f2_pack(__uint_as_float(r[2 + c][i]), __uint_as_float(r[2 + c][i + 1])), bu);
            silu_mul2(x, u, g[i], g[i + 1]);
          }
        }
      }
      if constexpr (DBG) {
        if (live) store_dbg32(dbg + row * n_out + n, g);
      }
      uint32_t w[6];
      const uint32_t sc = quant_block32(g, w);
      scale_word |= sc << (8 * c);
      if ((c & 1) == 0) {
#pragma unroll
        for (int i = 0; i < 6; ++i) wprev[i] = w[i];
        continue;
      }
      // two blocks' codes (48 bytes of the row) into the warp's slot, 48-byte rows:
      // 16-byte group 3 lane + j of the slot, distinct for eight consecutive lanes,
      // so the writes take the minimum wavefronts; then one TMA store of the
      // 32-row x 48-byte box
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      uint4* srow = reinterpret_cast<uint4*>(e.ostage + lane * kCodesBoxBytes);
      srow[0] = make_uint4(wprev[0], wprev[1], wprev[2], wprev[3]);
      srow[1] = make_uint4(wprev[4], wprev[5], w[0], w[1]);
      srow[2] = make_uint4(w[2], w[3], w[4], w[5]);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0 && row0 < m_total) {
        tma_store_2d(e.tmap_out, e.ostage, (n - 32) / 4 * 3, static_cast<int32_t>(row0));
        bulk_commit_group();
      }
    }
    // padding rows of the last row tile get zero scales; a row tile past the
    // last one (second half of the last pair) has no scale storage at all
    if (!live) scale_word = 0;
    if (mb < num_m) {
      uint8_t* sw = out_scales + scale_word_offset(row, col0 / kAtomK, n_out) + (col0 % kAtomK) / 32;
      if constexpr (kBlocks == 4)
        *reinterpret_cast<uint32_t*>(sw) = scale_word;
      else
        *reinterpret_cast<uint16_t*>(sw) = static_cast<uint16_t>(scale_word);
    }
  }
  return true;
}

// The warps of column group 1 during a half tile: nothing to drain; they release
// the accumulator (the barrier counts every epilogue warp) once it is full.
__device__ __forceinline__ bool epilogue_skip(SharedStorage& s, const EpiCtx& e, uint32_t& acc_phase,
                                              volatile int* abort_flag) {
  int ok = 0;
  if (e.lane == 0) ok = wait_bounded(&s.tmem_full, acc_phase, abort_flag, kErrWaitEpilogue) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  tc_fence_after();
  tc_fence_before();
  __syncwarp();
  if (e.lane == 0) mbar_arrive_remote_relaxed(e.tmem_empty_leader);
  acc_phase ^= 1u;
  return true;
}

template <int EPI, bool DBG, bool SPLIT, bool HALF>
__device__ __forceinline__ void run_epilogue(SharedStorage& s, uint32_t tmem, int warp, int lane, const Plan& pl,
                                             const CUtensorMap* tmap_out, const CUtensorMap* tmap_res, int cluster,
                                             int rank, int num_m,
                                             int m_total, int n_total,
                                             const uint16_t* __restrict__ bias, const uint16_t* __restrict__ gate,
                                             const uint16_t* residual, void* out, uint8_t* __restrict__ out_scales,
                                             float* __restrict__ dbg, volatile int* abort_flag) {
  EpiCtx e;
  e.warp = warp;
  e.lane = lane;
  e.q = warp & 3;           // tensor-memory lane quadrant this warp may access
  e.h = (warp - 2) >> 2;    // column group of the 256-wide tile
  e.rank = rank;
  e.cluster = cluster;
  e.num_m = num_m;
  e.m_total = m_total;
  e.n_total = n_total;
  e.n_out = (EPI == kEpiSwiglu) ? n_total / 2 : n_total;
  e.tmem = tmem;
  // the accumulator is released to the leader CTA's barrier (both CTAs' warps count)
  e.tmem_empty_leader = mapa_shared(smem_u32(&s.tmem_empty), 0);
  e.bw = s.bias_s[warp - 2];
  e.gw = s.gate_s[warp - 2];
  e.tmap_out = tmap_out;
  e.tmap_res = tmap_res;
  e.ostage = s.out_stage[warp - 2];
  e.res_bar = &s.res_full[warp - 2];
  e.res_phase = 0;
  uint32_t acc_phase = 0;
  // the split region first, in its own loop
  if constexpr (SPLIT) {
    Cursor cur = cursor_begin(pl, cluster);
    Unit u;
    while (cursor_next(pl, cur, u)) {
      int mb, nb;
      pair_tile(pl, u.tile, rank, &mb, &nb);
      if (!epilogue_tile<EPI, DBG, true>(s, e, mb, nb, nb * BN, acc_phase, pl, u, bias, gate, residual, out,
                                         out_scales, dbg, abort_flag))
        return;
    }
  }
  const Unit whole = {0, 0, 0};
  for (int p = (SPLIT ? pl.sk_tiles : 0) + cluster; p < (HALF ? pl.whole : pl.tiles); p += pl.clusters) {
    int mb, nb;
    pair_tile(pl, p, rank, &mb, &nb);
    if (!epilogue_tile<EPI, DBG, false>(s, e, mb, nb, nb * BN, acc_phase, pl, whole, bias, gate, residual, out,
                                        out_scales, dbg, abort_flag))
      return;
  }
  if constexpr (HALF) {
    if (cluster < 2 * pl.half_tiles) {
      int mb, nb;
      pair_tile(pl, pl.whole + cluster / 2, rank, &mb, &nb);
      if (e.h == 0)
        epilogue_tile<EPI, DBG, false>(s, e, mb, nb, nb * BN + (cluster % 2) * kHalfCols, acc_phase, pl, whole, bias,
                                       gate, residual, out, out_scales, dbg, abort_flag);
      else
        epilogue_skip(s, e, acc_phase, abort_flag);
    }
  }
}

// SPLIT: the launch divides its first sk_tiles tiles along K (a separate instance,
// so the whole-tile kernel carries none of that code). QA: the kernel quantizes A
// itself from BF16 (an extra warp; never with SPLIT). HALF: the last half_tiles
// tiles run as two 128-column halves on two pairs each (a separate instance too).
template <int EPI, bool DBG, bool SPLIT, bool QA, bool HALF>
__global__ void __launch_bounds__(QA ? kThreadsQa : kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_bh,
                   const __grid_constant__ CUtensorMap tmap_sa, const __grid_constant__ CUtensorMap tmap_sb,
                   const __grid_constant__ CUtensorMap tmap_out, const __grid_constant__ CUtensorMap tmap_res,
                   const uint16_t* __restrict__ bias, const uint16_t* __restrict__ gate, const uint16_t* residual,
                   void* out, uint8_t* __restrict__ out_scales, float* __restrict__ dbg, int m_total, int n_total,
                   int k_total, SplitArgs split, QaArgs qa) {
  static_assert(!(QA && SPLIT), "the in-kernel quantizer runs without the split tail");
  static_assert(!(HALF && (SPLIT || DBG || EPI == kEpiSwiglu)), "half tiles: whole-tile epilogues without debug output");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  SharedStorage& s =
      *reinterpret_cast<SharedStorage*>(smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr));
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int num_n = n_total / BN;
  const int num_m = (m_total + BM - 1) / BM;
  Plan plan;
  plan.num_n = num_n;
  plan.tiles = ((num_m + kPair - 1) / kPair) * num_n;
  plan.kblocks = k_total / BK;
  plan.clusters = static_cast<int>(cluster_count_x());
  plan.sk_tiles = split.sk_tiles;
  plan.half_tiles = HALF ? split.half_tiles : 0;
  plan.whole = plan.tiles - plan.half_tiles;
  plan.partial = split.partial;
  plan.arrivals = split.arrivals;
  const int cluster = static_cast<int>(cluster_id_x());
  const int rank = static_cast<int>(cluster_ctarank());

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
      mbar_init(&s.sfready[i], 1);
    }
    mbar_init(&s.tmem_full, 1);
    mbar_init(&s.tmem_empty, kPair * kEpiWarps);
    mbar_init(&s.drain, 1);
    for (int i = 0; i < kEpiWarps; ++i) mbar_init(&s.res_full[i], 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s.tmem_base, kTmemCols);  // both CTAs' warp 1 take part
    tmem_relinquish_pair();
    tc_fence_before();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    if (HALF) prefetch_tensormap(&tmap_bh);
    prefetch_tensormap(&tmap_sa);
    prefetch_tensormap(&tmap_sb);
    prefetch_tensormap(&tmap_out);
    if (EPI == kEpiGateRes) prefetch_tensormap(&tmap_res);
  }
  // both CTAs' barriers and tensor memory exist before either touches the other's
  cluster_sync();
  tc_fence_after();
  // the prologue above overlapped the previous kernel's tail; operands, bias and
  // outputs are touched only once it has completed
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    if (lane == 0)
      run_producer<SPLIT, QA, HALF>(s, &tmap_a, &tmap_b, &tmap_bh, &tmap_sa, &tmap_sb, plan, cluster, rank,
                                    EPI == kEpiSwiglu, n_total / 2, qa, num_m, abort_flag);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) run_mma<SPLIT, HALF>(s, tmem, plan, cluster, abort_flag);
  } else if (warp == 2 + kEpiWarps) {
    if (lane == 0 && rank == 0) run_scales<SPLIT, HALF>(s, tmem, plan, cluster, abort_flag);
  } else if (QA && warp == kQaWarp) {
    run_quantizer(qa, m_total, k_total, lane);
  } else {
    run_epilogue<EPI, DBG, SPLIT, HALF>(s, tmem, warp, lane, plan, &tmap_out, &tmap_res, cluster, rank, num_m,
                                        m_total, n_total,
                                        bias,
                                  gate, residual, out, out_scales, dbg, abort_flag);
    // the stores' writes are complete (and their shared sources read) before the
    // CTA leaves, also after a wait gave up
    if (lane == 0) bulk_wait_all();
  }
  __syncwarp();
  tc_fence_before();
  // neither CTA leaves (or frees tensor memory) while its peer may still touch it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map over packed 6-bit codes [rows][k]: 16U6 groups, box {128 codes, box_rows}.
static bool make_codes_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t k, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 4 * 3)};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B, 2, const_cast<void*>(codes), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor maps over the tiled scales, one 512-byte atom = 128 uint32 per box row.
// A: atoms [row tile][K step] as a 2-D [atoms][128]; box = one atom.
// B: [row tile][K step][128] as 3-D; box = the two atoms of one 256-row N tile, or
// (stacked gate/up weight) one atom, loaded once for the gate and once for the up rows.
static bool make_scale_maps(CUtensorMap* sa, CUtensorMap* sb, const void* a_scales, const void* b_scales, int64_t m,
                            int64_t n, int64_t k, uint32_t b_box_groups) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t kblocks = static_cast<cuuint64_t>(k / BK);
  std::memset(sa, 0, sizeof(*sa));
  std::memset(sb, 0, sizeof(*sb));
  cuuint64_t adims[2] = {128, static_cast<cuuint64_t>((m + BM - 1) / BM) * kblocks};
  cuuint64_t astr[1] = {kAtomBytes};
  cuuint32_t abox[2] = {128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(sa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(a_scales), adims, astr, abox, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  cuuint64_t bdims[3] = {128, kblocks, static_cast<cuuint64_t>(n / 128)};
  cuuint64_t bstr[2] = {kAtomBytes, kblocks * kAtomBytes};
  cuuint32_t bbox[3] = {128, 1, b_box_groups};
  r = fn(sb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(b_scales), bdims, bstr, bbox, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over a BF16 [m][n] matrix in the epilogues' boxes: 32 columns x 32 rows
// (one epilogue warp's block), 64-byte swizzle. The output's, for the TMA stores,
// and kEpiGateRes's residual, for its TMA loads.
static bool make_bf16_out_map(CUtensorMap* map, void* out, int64_t m, int64_t n) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(n) * 2};
  cuuint32_t box[2] = {kOutBoxCols, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over packed 6-bit output codes [m][w] (3 w / 4 bytes a row) for the
// requantizing epilogues' TMA stores: box 48 bytes (two MX blocks) x 32 rows.
static bool make_codes_out_map(CUtensorMap* map, void* codes, int64_t m, int64_t w) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  std::memset(map, 0, sizeof(*map));
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(w / 4 * 3), static_cast<cuuint64_t>(m)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(w / 4 * 3)};
  cuuint32_t box[2] = {kCodesBoxBytes, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, codes, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Per-device caches of the kernel attribute and of the co-resident cluster count,
// filled on a device's first call (any thread may fill them). The attribute belongs
// to the context, so it is set again when the device's context has changed (a new
// primary context after cudaDeviceReset).
template <int EPI, bool DBG, bool SPLIT, bool QA, bool HALF>
static cudaError_t max_clusters(int dev, cudaLaunchConfig_t cfg, int* clusters) {
  auto kern = mx_gemm_kernel<EPI, DBG, SPLIT, QA, HALF>;
  static std::atomic<unsigned long long> configured[64];   // context ID + 1 the attribute was set in; 0: none
  static std::atomic<int> cached[64];
  const bool cacheable = dev >= 0 && dev < 64;
  unsigned long long ctx = 0;
  if (!cacheable || !current_context_id(&ctx) || configured[dev].load(std::memory_order_acquire) != ctx + 1) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    if (cacheable && current_context_id(&ctx)) configured[dev].store(ctx + 1, std::memory_order_release);
  }
  int n = cacheable ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    cfg.gridDim = dim3(kPair * 64, 1, 1);
    cfg.numAttrs = 1;  // the cluster shape only
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorLaunchOutOfResources;
    if (cacheable) cached[dev].store(n, std::memory_order_relaxed);
  }
  *clusters = n;
  return cudaSuccess;
}

template <int EPI, bool DBG, bool QA>
static cudaError_t launch_instance(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
                                   const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& tout,
                                   const CUtensorMap& tres, const GemmArgs& a, cudaStream_t stream) {
  constexpr bool kHalvesOk = !DBG && EPI != kEpiSwiglu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel may start while the previous one in
  // the stream finishes; it waits (griddepcontrol.wait) before touching memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(QA ? kThreadsQa : kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int clusters = 0;
  e = max_clusters<EPI, DBG, false, QA, false>(dev, cfg, &clusters);
  if (e != cudaSuccess) return e;
  // as many CTA pairs as are co-resident (one CTA per SM), at most one per tile or half tile
  const GemmPlan plan =
      plan_gemm(a.m, a.n, a.k, clusters, QA ? nullptr : a.workspace, QA ? 0 : a.workspace_bytes, kHalvesOk);
  SplitArgs split = {};
  split.half_tiles = plan.half_tiles;
  if (plan.sk_tiles > 0) {
    split.sk_tiles = plan.sk_tiles;
    split.arrivals = static_cast<unsigned*>(a.workspace);
    split.partial = reinterpret_cast<float4*>(static_cast<uint8_t*>(a.workspace) + kArrivalsBytes);
  }
  QaArgs qa = {};
  if constexpr (QA) {
    qa.x = static_cast<const uint16_t*>(a.x);
    qa.ld_x = a.ld_x;
    qa.codes = static_cast<uint8_t*>(const_cast<void*>(a.a_codes));
    qa.scales = static_cast<uint8_t*>(const_cast<void*>(a.a_scales));
    qa.ready = a.ready;
    qa.first_block = static_cast<int>(a.lead_rows / 128);
    // counter word 0 is the quantizer warps' work counter: block 0 must be a leading one
    if (qa.first_block < 1) return cudaErrorInvalidValue;
    qa.strips = static_cast<int>(qa_strips(a.k));
    qa.wide = (reinterpret_cast<uintptr_t>(a.x) % 32 == 0 && a.ld_x % 16 == 0) ? 1 : 0;
  }
  cfg.gridDim = dim3(kPair * plan.clusters, 1, 1);
  // the split and half-tile instances have the same resources; their attribute is
  // set on first use
  int same = clusters;
  decltype(&mx_gemm_kernel<EPI, DBG, false, QA, false>) kern = mx_gemm_kernel<EPI, DBG, false, QA, false>;
  if constexpr (!QA) {
    if (plan.sk_tiles > 0) {
      e = max_clusters<EPI, DBG, true, false, false>(dev, cfg, &same);
      kern = mx_gemm_kernel<EPI, DBG, true, false, false>;
    }
  }
  if constexpr (kHalvesOk) {
    if (plan.half_tiles > 0) {
      e = max_clusters<EPI, DBG, false, QA, true>(dev, cfg, &same);
      kern = mx_gemm_kernel<EPI, DBG, false, QA, true>;
    }
  }
  if (e != cudaSuccess) return e;
  if (same != clusters) return cudaErrorLaunchOutOfResources;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tbh, tsa, tsb, tout, tres, static_cast<const uint16_t*>(a.bias),
                         static_cast<const uint16_t*>(a.gate), static_cast<const uint16_t*>(a.residual), a.out,
                         static_cast<uint8_t*>(a.out_scales), a.debug_prequant, static_cast<int>(a.m),
                         static_cast<int>(a.n), static_cast<int>(a.k), split, qa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, cudaStream_t stream, bool* encode_failed) {
  *encode_failed = false;
  CUtensorMap ta, tb, tbh, tsa, tsb, tout, tres;
  const bool bf16_out = a.epilogue == kEpiBf16 || a.epilogue == kEpiGateRes;
  const int64_t w_out = a.epilogue == kEpiSwiglu ? a.n / 2 : a.n;
  if (!make_codes_map(&ta, a.a_codes, a.m, a.k, BM) ||
      !make_codes_map(&tb, a.b_codes, a.n, a.k, kBHalfRows) ||
      !make_codes_map(&tbh, a.b_codes, a.n, a.k, kHalfCols / kPair) ||
      !make_scale_maps(&tsa, &tsb, a.a_scales, a.b_scales, a.m, a.n, a.k, a.epilogue == kEpiSwiglu ? 1u : 2u) ||
      !(bf16_out ? make_bf16_out_map(&tout, a.out, a.m, a.n) : make_codes_out_map(&tout, a.out, a.m, w_out)) ||
      // kEpiGateRes reads the residual [M][N] in the output's boxes; other epilogues
      // pass the output's map, unused
      !(a.epilogue == kEpiGateRes ? make_bf16_out_map(&tres, const_cast<void*>(a.residual), a.m, a.n)
                                  : (tres = tout, true))) {
    *encode_failed = true;
    return cudaSuccess;
  }
  (void)num_sms;
  const bool dbg = a.debug_prequant != nullptr;
  if (a.x != nullptr) {
    // the in-kernel quantizer: no debug output, no split tail
    if (dbg) return cudaErrorInvalidValue;
    switch (a.epilogue) {
      case kEpiBf16: return launch_instance<kEpiBf16, false, true>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
      case kEpiGelu: return launch_instance<kEpiGelu, false, true>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
      case kEpiSwiglu: return launch_instance<kEpiSwiglu, false, true>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
      case kEpiGateRes: return launch_instance<kEpiGateRes, false, true>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.epilogue) {
    case kEpiBf16: return launch_instance<kEpiBf16, false, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
    case kEpiGelu:
      return dbg ? launch_instance<kEpiGelu, true, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream)
                 : launch_instance<kEpiGelu, false, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
    case kEpiSwiglu:
      return dbg ? launch_instance<kEpiSwiglu, true, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream)
                 : launch_instance<kEpiSwiglu, false, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
    case kEpiGateRes: return launch_instance<kEpiGateRes, false, false>(ta, tb, tbh, tsa, tsb, tout, tres, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_max_clusters(int* clusters) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return max_clusters<kEpiBf16, false, false, false, false>(dev, cfg, clusters);
}

// A wait that nothing will ever satisfy: it must give up after the bound, set
// its error bit and let the kernel return with the context intact.
__global__ void wait_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(&bar, 0, &abort_flag, kErrSelfTest);
}

cudaError_t launch_wait_selftest(cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t read_device_error(unsigned* flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_error_word, sizeof(unsigned));
  if (e != cudaSuccess || !clear) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
}

}  // namespace mxk
