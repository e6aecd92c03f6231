// The tcgen05 GEMM mainloop shared by the projections of the chunk step:
//   D[256 x BN] = A[256 x K] . B[BN x K]^T,  bf16 operands, fp32 accumulators.
// Two 128-row tcgen05.mma halves share every B tile (half the L2 feed per
// flop of a 128-row tile); TMA fills a 3-stage ring of 128-byte-swizzled
// tiles.  Block roles (384 threads): warp 0 TMA producer, warp 1 TMEM
// allocation and MMA issue, warps 4-11 the caller's epilogue (warps 2-3 idle).
// Accumulator rows 0-127 live in TMEM columns [0, BN), rows 128-255 in
// [BN, 2 BN).  Every wait is bounded; a timeout is recorded in the device
// error word with the caller's flag bit.
#pragma once

#include "common.h"
#include "ptx.cuh"

namespace savgb {
namespace gemm {

constexpr int kThreads = 384;
constexpr int kBM = 256;
constexpr int kBK = 64;
constexpr int kStages = 3;

template <int BN>
struct Layout {
  static constexpr int kAHalf = 128 * kBK * 2;  // 16 KiB
  static constexpr int kABytes = 2 * kAHalf;
  static constexpr int kBBytes = BN * kBK * 2;  // 16 or 32 KiB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBar = kStages * kStageBytes;
  static constexpr int kMisc = kBar + (2 * kStages + 2) * 8;
  static constexpr int kExtra = kMisc + 16;  // start of the epilogue's own shared memory
  static constexpr int kDynSmem = kExtra + 1024;
  static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
  static_assert(8 * 4096 <= kBar, "epilogue staging must fit in the ring");
};

struct Ctx {
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* drain;
  volatile int* abort;
  uint32_t tmem;
};

__device__ __forceinline__ void give_up(DeviceErrorWord* err, volatile int* abort, unsigned flag,
                                        unsigned code) {
  if (atomicExch(const_cast<int*>(abort), 1) == 0) {
    atomicOr(&err->flags, flag);
    atomicCAS(&err->where, 0u, code);
  }
}

// Barriers, abort flag and the 2*BN TMEM columns; every thread calls it.
template <int BN>
__device__ __forceinline__ Ctx setup(uint8_t* smem_raw, const CUtensorMap* map_a, const CUtensorMap* map_b) {
  using L = Layout<BN>;
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  Ctx c;
  c.smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  c.full = reinterpret_cast<uint64_t*>(c.smem + L::kBar);
  c.empty = c.full + kStages;
  c.acc_full = c.empty + kStages;
  c.drain = c.acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.smem + L::kMisc);
  c.abort = reinterpret_cast<volatile int*>(c.smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(&c.full[s], 1);
      dev::mbar_init(&c.empty[s], 1);
    }
    dev::mbar_init(c.acc_full, 1);
    dev::mbar_init(c.drain, 1);
    *c.abort = 0;
    dev::fence_barrier_init();
  }
  if (warp == 1) {
    dev::tmem_alloc(tmem_slot, 2 * BN);
    dev::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    dev::tma_prefetch_desc(map_a);
    dev::tma_prefetch_desc(map_b);
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  c.tmem = *tmem_slot;
  return c;
}

// Warp 0, lane 0: streams the k-blocks of A (two 128-row halves) and B.
template <int BN>
__device__ __forceinline__ void produce(const Ctx& c, const CUtensorMap* map_a, const CUtensorMap* map_b, int m0,
                                        int n0, int kb_count, DeviceErrorWord* err, unsigned flag) {
  using L = Layout<BN>;
  int issued = 0;
  for (int kb = 0; kb < kb_count; ++kb) {
    const int st = kb % kStages;
    const uint32_t use = kb / kStages;
    if (kb >= kStages && !dev::mbar_wait(&c.empty[st], (use - 1) & 1, c.abort)) {
      give_up(err, c.abort, flag, 1);
      break;
    }
    uint8_t* sa = c.smem + st * L::kStageBytes;
    dev::mbar_arrive_expect_tx(&c.full[st], L::kStageBytes);
    dev::tma_load_2d(sa, map_a, &c.full[st], kb * kBK, m0);
    dev::tma_load_2d(sa + L::kAHalf, map_a, &c.full[st], kb * kBK, m0 + 128);
    dev::tma_load_2d(sa + L::kABytes, map_b, &c.full[st], kb * kBK, n0);
    issued = kb + 1;
  }
  volatile int never = 0;
  for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
    dev::mbar_wait(&c.full[t % kStages], (t / kStages) & 1, &never);
}

// Warp 1, lane 0: issues the MMAs, then signals acc_full; drains before exit.
template <int BN>
__device__ __forceinline__ void mma(const Ctx& c, int kb_count, DeviceErrorWord* err, unsigned flag) {
  // the whole warp runs the loop (warp-uniform state); one elected lane
  // issues the MMAs and commits
  using L = Layout<BN>;
  const bool leader = dev::elect_one();
  constexpr uint32_t idesc = dev::idesc_bf16_f32(128, BN, false, false);
  const uint64_t d0 = dev::sdesc_sw128(dev::smem_u32(c.smem), 16, 1024);
  bool ok = true;
  for (int kb = 0; kb < kb_count; ++kb) {
    const int st = kb % kStages;
    if (!__all_sync(0xffffffffu, dev::mbar_wait(&c.full[st], (kb / kStages) & 1, c.abort))) {
      if (leader) give_up(err, c.abort, flag, 2);
      ok = false;
      break;
    }
    dev::tc_fence_after();
    if (leader) {
      const uint64_t ds = d0 + static_cast<uint32_t>((st * L::kStageBytes) >> 4);
      #pragma unroll
      for (int k = 0; k < kBK / 16; ++k) {
        const uint32_t koff = (k * 32) >> 4;
        const uint64_t bd = ds + ((L::kABytes >> 4) + koff);
        dev::mma_ss(c.tmem, ds + koff, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        dev::mma_ss(c.tmem + BN, ds + ((L::kAHalf >> 4) + koff), bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      dev::mma_commit(&c.empty[st]);
    }
  }
  if (leader) {
    if (ok) dev::mma_commit(c.acc_full);
    dev::mma_commit(c.drain);
  }
  __syncwarp();
  volatile int never = 0;
  dev::mbar_wait(c.drain, 0, &never);
}

// Epilogue warps: wait for the accumulators (every lane polls, a vote keeps
// the warp on one path); false on abort.
__device__ __forceinline__ bool wait_acc(const Ctx& c, DeviceErrorWord* err, unsigned flag) {
  const bool ok = __all_sync(0xffffffffu, dev::mbar_wait(c.acc_full, 0, c.abort));
  if (ok) dev::tc_fence_after();
  else give_up(err, c.abort, flag, 3);
  return ok;
}

// Every thread, at the end.
template <int BN>
__device__ __forceinline__ void teardown(const Ctx& c) {
  dev::tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc(c.tmem, 2 * BN);
  }
}

}  // namespace gemm
}  // namespace savgb
