// The persistent CTA-pair tcgen05 GEMM mainloop shared by the projections of
// the chunk step (W_o with the Euler update, and the QKV projection of a
// block step):  D[256 x 256] tiles of  A[M x K] . B[N x K]^T,  bf16 operands,
// fp32 accumulators, over clusters of two CTAs on two SMs.
//
// tcgen05.mma.cta_group::2 with M = 256 and N = 256: each CTA holds 128 rows
// of A and 128 of the 256 rows of the B tile in a ring of TMA-filled,
// 128-byte-swizzled stages, and two 128 x 256 fp32 accumulators in TMEM (all
// 512 columns), so the caller's epilogue of one tile reads one accumulator
// while the MMAs of the cluster's next tile fill the other.
//   warp 0      TMA producer of this CTA's A rows and B half
//   warp 1      TMEM allocation (both CTAs); the even CTA's warp runs the MMA
//               issue loop, one elected lane issues and commits to both CTAs
//   warp 2      (odd CTA) relays "stage full" to the even CTA's barrier
//   warps 4-11  the caller's epilogue: warp -> 32 rows (its TMEM lane
//               quadrant) x 128 columns (one half of the tile)
// Tiles are taken round robin: cluster c computes tiles c, c + clusters, ...;
// tile t covers rows (t / n_tiles_n) * 256 and columns (t % n_tiles_n) * 256.
// Every wait is bounded; a timeout is recorded in the device error word with
// the caller's flag bit, and each role leaves its loop.
//
// Shared memory: STAGES ring | epilogue staging (4 KiB per epilogue warp) |
// barriers | misc | the caller's extra bytes.
#pragma once

#include "common.h"
#include "ptx.cuh"

namespace savgb {
namespace gemm_pair {

constexpr int kThreads = 384;
constexpr int kBK = 64;
constexpr int kTile = 256;
constexpr int kABytes = 128 * kBK * 2;  // 16 KiB: this CTA's 128 rows of A
constexpr int kBBytes = 128 * kBK * 2;  // 16 KiB: this CTA's 128 rows of the B tile
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kWarpStaging = 4096;      // per epilogue warp
constexpr int kStagingBytes = 8 * kWarpStaging;

// EXTRA_BARS: the caller's own barriers (count 1 each, in this CTA).
template <int STAGES, int EXTRA_BARS>
struct Layout {
  static constexpr int kStages = STAGES;
  static constexpr int kStaging = STAGES * kStageBytes;
  static constexpr int kBar = kStaging + kStagingBytes;
  static constexpr int kFull = 0, kEmpty = STAGES, kAccFull = 2 * STAGES, kAccEmpty = kAccFull + 2;
  static constexpr int kDrain = kAccEmpty + 2;
  static constexpr int kExtraBar = kDrain + 1;
  static constexpr int kNumBars = kExtraBar + EXTRA_BARS;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kExtra = (kMisc + 16 + 127) / 128 * 128;  // start of the caller's extra bytes
  static constexpr int kDynSmem = kExtra + 1024;                 // + the caller's extra bytes
};

struct Ctx {
  uint8_t* smem;
  uint64_t* bars;
  volatile int* abort;
  uint32_t tmem;
  uint32_t rank;  // in the cluster
  bool leader;    // the even CTA
  int cluster, n_clusters;
};

// The error word and flag of the caller, and the failure-path test hook: the
// k-block iteration whose relay the odd CTA of cluster 0 leaves out (< 0:
// none) and the limit of every wait.
struct Hook {
  DeviceErrorWord* err;
  unsigned flag;
  int fault_iter;
  uint64_t limit_ns;
};

__device__ __forceinline__ void give_up(const Hook& h, volatile int* abort, unsigned code) {
  if (atomicExch(const_cast<int*>(abort), 1) == 0) {
    atomicOr(&h.err->flags, h.flag);
    atomicCAS(&h.err->where, 0u, code);
  }
}

// Every thread of both CTAs: barriers, the caller's barriers, TMEM.
template <class L>
__device__ __forceinline__ Ctx setup(uint8_t* smem_raw, const CUtensorMap* map_a, const CUtensorMap* map_b,
                                     const CUtensorMap* map_c) {
  Ctx c;
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  c.smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  c.bars = reinterpret_cast<uint64_t*>(c.smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.smem + L::kMisc);
  c.abort = reinterpret_cast<volatile int*>(c.smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  c.rank = dev::cluster_rank();
  c.leader = c.rank == 0;
  c.cluster = static_cast<int>(blockIdx.x >> 1);
  c.n_clusters = static_cast<int>(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      dev::mbar_init(&c.bars[L::kFull + s], c.leader ? 2 : 1);  // the even CTA's: its own load + the odd CTA's relay
      dev::mbar_init(&c.bars[L::kEmpty + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&c.bars[L::kAccFull + b], 1);
      dev::mbar_init(&c.bars[L::kAccEmpty + b], 16);  // the 8 epilogue warps of both CTAs (even CTA's copy)
    }
    dev::mbar_init(&c.bars[L::kDrain], 1);
    for (int i = L::kExtraBar; i < L::kNumBars; ++i) dev::mbar_init(&c.bars[i], 1);
    *c.abort = 0;
    dev::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    dev::tma_prefetch_desc(map_a);
    dev::tma_prefetch_desc(map_b);
    if (map_c) dev::tma_prefetch_desc(map_c);
  }
  __syncthreads();
  dev::cluster_sync();  // both CTAs' barriers exist before any remote arrive
  if (warp == 1) {
    dev::tmem_alloc_pair(tmem_slot, 512);
    dev::tmem_relinquish_pair();
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::cluster_sync();
  dev::tc_fence_after();
  c.tmem = *tmem_slot;
  return c;
}

// Warp 0, lane 0 of both CTAs: this CTA's A rows and B half of every k-block
// of the cluster's tiles, then waits until every copy it issued has landed.
template <class L>
__device__ __forceinline__ void produce(const Ctx& c, const Hook& h, const CUtensorMap* map_a,
                                        const CUtensorMap* map_b, int n_tiles_n, int n_tiles, int kb_count) {
  uint32_t it = 0;
  bool ok = true;
  for (int t = c.cluster; t < n_tiles && ok; t += c.n_clusters) {
    const int m0 = (t / n_tiles_n) * kTile + static_cast<int>(c.rank) * 128;
    const int nb = (t % n_tiles_n) * kTile + static_cast<int>(c.rank) * 128;
    for (int kb = 0; kb < kb_count; ++kb, ++it) {
      const int st = static_cast<int>(it % L::kStages);
      const uint32_t use = it / L::kStages;
      if (use > 0 && !dev::mbar_wait(&c.bars[L::kEmpty + st], (use - 1) & 1, c.abort, h.limit_ns)) {
        give_up(h, c.abort, 11);
        ok = false;
        break;
      }
      uint8_t* sa = c.smem + st * kStageBytes;
      dev::mbar_arrive_expect_tx(&c.bars[L::kFull + st], kStageBytes);
      dev::tma_load_2d(sa, map_a, &c.bars[L::kFull + st], kb * kBK, m0);
      dev::tma_load_2d(sa + kABytes, map_b, &c.bars[L::kFull + st], kb * kBK, nb);
    }
  }
  volatile int never = 0;
  const uint32_t first = it > static_cast<uint32_t>(L::kStages) ? it - L::kStages : 0;
  for (uint32_t t = first; t < it; ++t) {
    if (c.leader) dev::mbar_wait_cluster(&c.bars[L::kFull + t % L::kStages], (t / L::kStages) & 1, &never, h.limit_ns);
    else dev::mbar_wait(&c.bars[L::kFull + t % L::kStages], (t / L::kStages) & 1, &never, h.limit_ns);
  }
}

// Warp 1 of the even CTA: the whole warp runs the loop (warp-uniform state),
// one elected lane issues the MMAs and commits to both CTAs' barriers; every
// MMA has completed before it returns.
template <class L>
__device__ __forceinline__ void mma(const Ctx& c, const Hook& h, int n_tiles, int kb_count) {
  const bool issuer = dev::elect_one();
  constexpr uint32_t idesc = dev::idesc_bf16_f32(256, 256, false, false);
  const uint64_t d0 = dev::sdesc_sw128(dev::smem_u32(c.smem), 16, 1024);
  uint32_t it = 0;
  int tile_i = 0;
  bool ok = true;
  for (int t = c.cluster; t < n_tiles && ok; t += c.n_clusters, ++tile_i) {
    const int buf = tile_i & 1;
    const uint32_t buse = static_cast<uint32_t>(tile_i >> 1);
    if (buse > 0 &&
        !__all_sync(0xffffffffu, dev::mbar_wait_cluster(&c.bars[L::kAccEmpty + buf], (buse - 1) & 1, c.abort,
                                                        h.limit_ns))) {
      if (issuer) give_up(h, c.abort, 12);
      break;
    }
    dev::tc_fence_after();
    const uint32_t d = c.tmem + static_cast<uint32_t>(buf * 256);
    for (int kb = 0; kb < kb_count; ++kb, ++it) {
      const int st = static_cast<int>(it % L::kStages);
      if (!__all_sync(0xffffffffu,
                      dev::mbar_wait(&c.bars[L::kFull + st], (it / L::kStages) & 1, c.abort, h.limit_ns))) {
        if (issuer) give_up(h, c.abort, 13);
        ok = false;
        break;
      }
      dev::tc_fence_after();
      if (issuer) {
        const uint64_t ds = d0 + static_cast<uint32_t>((st * kStageBytes) >> 4);
        #pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint32_t koff = (k * 32) >> 4;
          dev::mma_ss_pair(d, ds + koff, ds + ((kABytes >> 4) + koff), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        dev::mma_commit_pair(&c.bars[L::kEmpty + st], 3);
      }
    }
    if (ok && issuer) dev::mma_commit_pair(&c.bars[L::kAccFull + buf], 3);
  }
  // every MMA has completed before TMEM is released
  if (issuer) dev::mma_commit_pair(&c.bars[L::kDrain], 1);
  __syncwarp();
  volatile int never = 0;
  dev::mbar_wait(&c.bars[L::kDrain], 0, &never, h.limit_ns);
}

// Warp 2, lane 0 of the odd CTA: forwards "stage full" to the even CTA.
template <class L>
__device__ __forceinline__ void relay(const Ctx& c, const Hook& h, int n_tiles, int kb_count) {
  const uint32_t full0 = dev::mapa_shared(&c.bars[L::kFull], 0);
  // test hook: the first cluster leaves one relay out (fault_iter < 0: never)
  const int64_t skip = c.cluster == 0 ? h.fault_iter : -1;
  uint32_t it = 0;
  bool ok = true;
  for (int t = c.cluster; t < n_tiles && ok; t += c.n_clusters) {
    for (int kb = 0; kb < kb_count; ++kb, ++it) {
      const int st = static_cast<int>(it % L::kStages);
      if (!dev::mbar_wait(&c.bars[L::kFull + st], (it / L::kStages) & 1, c.abort, h.limit_ns)) {
        give_up(h, c.abort, 14);
        ok = false;
        break;
      }
      // relaxed: the TMA completion just observed already placed the data; a
      // release arrive at cluster scope held this thread ~0.8 us per stage and
      // throttled the whole pipeline to half speed
      if (static_cast<int64_t>(it) != skip) dev::mbar_arrive_cluster_relaxed(full0 + static_cast<uint32_t>(st * 8));
    }
  }
}

// Epilogue warps: the accumulator of the cluster's tile_i-th tile is ready
// (every lane polls, a vote keeps the warp on one path); false on abort.
template <class L>
__device__ __forceinline__ bool acc_wait(const Ctx& c, const Hook& h, int tile_i) {
  const bool ok = __all_sync(0xffffffffu, dev::mbar_wait_cluster(&c.bars[L::kAccFull + (tile_i & 1)],
                                                                 (tile_i >> 1) & 1, c.abort, h.limit_ns));
  if (ok) dev::tc_fence_after();
  else give_up(h, c.abort, 15);
  return ok;
}

// Epilogue warps, after reading their part of the accumulator of tile_i.
template <class L>
__device__ __forceinline__ void acc_release(const Ctx& c, int tile_i) {
  const int buf = tile_i & 1;
  dev::tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (c.leader) dev::mbar_arrive(&c.bars[L::kAccEmpty + buf]);
    else dev::mbar_arrive_cluster(dev::mapa_shared(&c.bars[L::kAccEmpty + buf], 0));
  }
}

// Every thread of both CTAs, at the end: neither CTA leaves (or frees TMEM)
// while its peer may still use its shared memory or run pair MMAs.  Both CTAs
// reach these cluster barriers after a give-up too: every wait above is
// bounded and the drain makes the MMAs complete first.
__device__ __forceinline__ void teardown(const Ctx& c) {
  dev::tc_fence_before();
  __syncthreads();
  dev::cluster_sync();
  if ((threadIdx.x >> 5) == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc_pair(c.tmem, 512);
  }
  __syncthreads();
  dev::cluster_sync();
}

// The cluster count of one wave of a pair kernel: as many clusters as can be
// resident at once (cached per device by the caller).
template <typename Kernel>
int max_clusters(Kernel kernel, int sms, int smem, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * (sms / 2)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  SAVGB_CUDA(cudaOccupancyMaxActiveClusters(&n, kernel, &cfg));
  *out = n > 0 ? n : 1;
  return SAVGB_OK;
}

}  // namespace gemm_pair
}  // namespace savgb
