// Output projection + flow-matching Euler update on the sm_103a tensor cores.
//
//   v = O W_o^T (+ bias);  x <- x + dt * v
//
// The attention output is projected by W_o and taken as the velocity of the
// flow, then one explicit Euler step is applied to the state (HeyGen, "Avatar
// inference at scale", section "The underlying model architecture": a DiT
// trained with flow matching; section "The streaming framework and pipeline
// loop": a multi-step diffusion pass per chunk).
//
// One CTA computes a 256 x BN tile of v: two 128-row tcgen05.mma halves share
// every B (W_o) tile, so each byte fed from L2 does twice the work of a
// 128-row tile.  bf16 operands sit in 128-byte-swizzled shared memory fed by
// TMA through a 3-stage ring; the fp32 accumulators live in TMEM.  The
// epilogue reads them back, turns each 32 x 32 chunk around in shared memory
// and applies the Euler update to x (fp32, read-modify-write) with coalesced
// 128-byte row segments, so v never goes through global memory.
//   warp 0      TMA producer
//   warp 1      TMEM allocation; lane 0 issues the MMAs
//   warps 4-11  epilogue (warps 2-3 idle)
#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

namespace savgb {
namespace {

constexpr int kThreads = 384;
constexpr int kBM = 256;  // two 128-row MMA halves share every B tile
constexpr int kBK = 64;
constexpr int kStages = 3;

struct WoParams {
  int M, N, K;
  float dt;
  const float* bias;
  float* x;
  float* v_out;
  DeviceErrorWord* err;
};

template <int BN>
struct WoLayout {
  static constexpr int kAHalf = 128 * kBK * 2;  // 16 KiB
  static constexpr int kABytes = 2 * kAHalf;
  static constexpr int kBBytes = BN * kBK * 2;  // 16 or 32 KiB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBar = kStages * kStageBytes;
  static constexpr int kMisc = kBar + (2 * kStages + 2) * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kDynSmem <= 227 * 1024, "shared memory budget");
  static_assert(8 * 4096 <= kBar, "epilogue staging must fit in the ring");
};

__device__ __forceinline__ void give_up(const WoParams& p, volatile int* abort, unsigned code) {
  if (atomicExch(const_cast<int*>(abort), 1) == 0) {
    atomicOr(&p.err->flags, kErrGemmWait);
    atomicCAS(&p.err->where, 0u, 0x100u + code);
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    wo_euler_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b, const WoParams p) {
  using L = WoLayout<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * kBM;
  const int kb_count = (p.K + kBK - 1) / kBK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    dev::mbar_init(acc_full, 1);
    dev::mbar_init(drain, 1);
    *abort = 0;
    dev::fence_barrier_init();
  }
  if (warp == 1) {
    dev::tmem_alloc(tmem_slot, 2 * BN);
    dev::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    dev::tma_prefetch_desc(&map_a);
    dev::tma_prefetch_desc(&map_b);
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < kb_count; ++kb) {
        const int st = kb % kStages;
        const uint32_t use = kb / kStages;
        if (kb >= kStages && !dev::mbar_wait(&empty[st], (use - 1) & 1, abort)) {
          give_up(p, abort, 1);
          break;
        }
        uint8_t* sa = smem + st * L::kStageBytes;
        dev::mbar_arrive_expect_tx(&full[st], L::kStageBytes);
        dev::tma_load_2d(sa, &map_a, &full[st], kb * kBK, m0);
        dev::tma_load_2d(sa + L::kAHalf, &map_a, &full[st], kb * kBK, m0 + 128);
        dev::tma_load_2d(sa + L::kABytes, &map_b, &full[st], kb * kBK, n0);
        issued = kb + 1;
      }
      volatile int never = 0;
      for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
        dev::mbar_wait(&full[t % kStages], (t / kStages) & 1, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = dev::idesc_bf16_f32(128, BN, false, false);
      const uint64_t d0 = dev::sdesc_sw128(dev::smem_u32(smem), 16, 1024);
      bool ok = true;
      for (int kb = 0; kb < kb_count; ++kb) {
        const int st = kb % kStages;
        if (!dev::mbar_wait(&full[st], (kb / kStages) & 1, abort)) {
          give_up(p, abort, 2);
          ok = false;
          break;
        }
        dev::tc_fence_after();
        const uint64_t ds = d0 + static_cast<uint32_t>((st * L::kStageBytes) >> 4);
        #pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint32_t koff = (k * 32) >> 4;
          const uint64_t bd = ds + ((L::kABytes >> 4) + koff);
          dev::mma_ss(tmem, ds + koff, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          dev::mma_ss(tmem + BN, ds + ((L::kAHalf >> 4) + koff), bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        dev::mma_commit(&empty[st]);
      }
      if (ok) dev::mma_commit(acc_full);
      dev::mma_commit(drain);
      volatile int never = 0;
      dev::mbar_wait(drain, 0, &never);
    }
  } else if (warp >= 4) {
    // epilogue: warps 4-7 take rows 0-127 (accumulator columns [0, BN)),
    // warps 8-11 rows 128-255 ([BN, 2 BN)).  Each 32-row x 32-column chunk is
    // loaded from TMEM (one row per lane), turned around in shared memory and
    // applied to x with 8 lanes per 128-byte row segment (coalesced).
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row_base = m0 + half * 128 + quad * 32;
    // while the MMAs run, pull this warp's 32 rows of x (BN columns) into L2
    {
      const int m = row_base + lane;
      const int ncols = min(BN, p.N - n0);
      if (m < p.M && ncols > 0) dev::prefetch_l2(p.x + static_cast<int64_t>(m) * p.N + n0, ncols * 4);
    }
    bool ok = true;
    if (lane == 0) ok = dev::mbar_wait(acc_full, 0, abort);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
      dev::tc_fence_after();
      // the operand ring is idle once every MMA has completed: 4 KiB per warp
      float4* stage = reinterpret_cast<float4*>(smem + (warp - 4) * 4096);
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16) + half * BN;
      const float dt = p.dt;
      const int seg = lane & 7;
      #pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t acc[32];
        dev::tmem_ld32(t_row + c, acc);
        #pragma unroll
        for (int j = 0; j < 8; ++j)
          stage[lane * 8 + ((j + lane) & 7)] =
              make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                          __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
        __syncwarp();
        const int n = n0 + c + 4 * seg;
        float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.bias && n < p.N) bb = *reinterpret_cast<const float4*>(p.bias + n);
        // all eight loads of x first (the stores below could alias them as far
        // as the compiler knows), then the updates
        float4 xv[8];
        float4 v[8];
        #pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = 4 * k + (lane >> 3);
          const int m = row_base + r;
          v[k] = stage[r * 8 + ((seg + r) & 7)];
          if (m < p.M && n < p.N)  // N % 16 == 0: a group of 4 columns is all in or all out
            xv[k] = *reinterpret_cast<const float4*>(p.x + static_cast<int64_t>(m) * p.N + n);
        }
        #pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int m = row_base + 4 * k + (lane >> 3);
          if (m < p.M && n < p.N) {
            float4 u = v[k];
            u.x += bb.x; u.y += bb.y; u.z += bb.z; u.w += bb.w;
            float4 y = xv[k];
            y.x = fmaf(dt, u.x, y.x);
            y.y = fmaf(dt, u.y, y.y);
            y.z = fmaf(dt, u.z, y.z);
            y.w = fmaf(dt, u.w, y.w);
            *reinterpret_cast<float4*>(p.x + static_cast<int64_t>(m) * p.N + n) = y;
            if (p.v_out) *reinterpret_cast<float4*>(p.v_out + static_cast<int64_t>(m) * p.N + n) = u;
          }
        }
        __syncwarp();
      }
    } else {
      give_up(p, abort, 3);
    }
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, 2 * BN);
  }
}

template <int BN>
int launch_bn(const void* o, const void* w, const float* bias, float* x, int64_t M, int K, int N,
              float dt, float* v_out, cudaStream_t stream) {
  using L = WoLayout<BN>;
  static bool attr_done[64] = {false};
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (!attr_done[dev_id & 63]) {
    SAVGB_CUDA(cudaFuncSetAttribute(wo_euler_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::kDynSmem));
    attr_done[dev_id & 63] = true;
  }
  CUtensorMap ma, mb;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M};
  const uint64_t sa[1] = {(uint64_t)K * 2};
  const uint32_t ba[2] = {kBK, 128};
  int rc = encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N};
  const uint32_t bb[2] = {kBK, BN};
  rc = encode_tiled(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, db, sa, bb, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  WoParams p{(int)M, N, K, dt, bias, x, v_out, nullptr};
  if ((rc = error_word(&p.err))) return rc;
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + kBM - 1) / kBM));
  wo_euler_kernel<BN><<<grid, kThreads, L::kDynSmem, stream>>>(ma, mb, p);
  SAVGB_CUDA(cudaGetLastError());
  return SAVGB_OK;
}

}  // namespace

int validate_out_proj(const void* o, const void* w, const float* bias, const float* x, int64_t M,
                      int hid_in, int hid_out, const float* v_out) {
  if (!o || !w || !x) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: null o, w_o or x");
  if (!aligned16(o) || !aligned16(w) || !aligned16(x) || (bias && !aligned16(bias)) ||
      (v_out && !aligned16(v_out)))
    return fail(SAVGB_ERR_ALIGNMENT, "out_proj_euler_step: pointers must be 16-byte aligned");
  if (M < 1 || M > ((int64_t)1 << 31) - 1 - kBM) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: M must be in [1, 2^31)");
  if (hid_in < 8 || hid_in % 8) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hid_in must be a positive multiple of 8");
  if (hid_out < 16 || hid_out % 16) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hid_out must be a positive multiple of 16");
  if (hid_in > (1 << 24) || hid_out > (1 << 24)) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hidden size too large");
  return SAVGB_OK;
}

int launch_out_proj_euler(const void* o, const void* w, const float* bias, float* x, int64_t M,
                          int hid_in, int hid_out, float dt, float* v_out, cudaStream_t stream) {
  int rc = check_device(nullptr);
  if (rc) return rc;
  if (hid_out % 256 == 0)
    return launch_bn<256>(o, w, bias, x, M, hid_in, hid_out, dt, v_out, stream);
  return launch_bn<128>(o, w, bias, x, M, hid_in, hid_out, dt, v_out, stream);
}

}  // namespace savgb

extern "C" int out_proj_euler_step(const void* o, const void* w_o, const float* bias, float* x,
                                   int64_t M, int hid_in, int hid_out, float dt, float* v_out,
                                   void* stream) {
  using namespace savgb;
  clear_error();
  int rc = validate_out_proj(o, w_o, bias, x, M, hid_in, hid_out, v_out);
  if (rc) return rc;
  return launch_out_proj_euler(o, w_o, bias, x, M, hid_in, hid_out, dt, v_out,
                               static_cast<cudaStream_t>(stream));
}
