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
// Two kernels.  When only x is updated and the output width is a multiple of
// 256, a persistent CTA-pair kernel (below) computes 256 x 256 tiles with
// double-buffered accumulators, so each tile's Euler epilogue overlaps the
// next tile's MMAs.  Otherwise (other widths, or the velocity also written
// out) one CTA computes a 256 x BN tile of v: two 128-row tcgen05.mma halves share
// every B (W_o) tile, so each byte fed from L2 does twice the work of a
// 128-row tile.  bf16 operands sit in 128-byte-swizzled shared memory fed by
// TMA through a 3-stage ring; the fp32 accumulators live in TMEM.  The
// epilogue stages x through the (then idle) ring with tensor-map loads and
// stores, 32 x 32 fp32 chunks, several in flight per warp, and each thread
// applies the Euler update to its row with v straight from its TMEM lane, so
// v never goes through global memory.
// The mainloop (TMA producer, MMA issue, TMEM) is the shared 256-row GEMM of
// gemm_tc.cuh; warps 4-11 run the Euler epilogue.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.h"
#include "gemm_pair.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace savgb {
namespace {

struct WoParams {
  int M, N, K;
  float dt;
  const float* bias;
  float* x;
  float* v_out;
  DeviceErrorWord* err;
  // failure-path test hook of the CTA-pair kernel (savgb_arm_wait_fault):
  // k-block iteration whose relay the odd CTA of cluster 0 skips (-1: none),
  // and the limit of every wait of that kernel
  int fault_iter;
  uint64_t wait_limit_ns;
  // optional fp32 [M][N]: receives a copy of the updated x (the same tensor-map
  // stores, a second destination); x-only epilogues, not with v_out
  float* x_copy;
};

constexpr int kXChunk = 32;                   // columns of x per staged chunk
constexpr int kXChunkBytes = 32 * kXChunk * 4;  // a warp's 32 rows x 32 fp32 columns
constexpr int kXBufs = 4;                       // chunks of x in flight per warp

template <int BN>
__global__ void __launch_bounds__(gemm::kThreads, 1)
    wo_euler_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_xc, const WoParams p) {
  using L = gemm::Layout<BN>;
  static_assert(8 * kXBufs * kXChunkBytes <= L::kBar, "x staging must fit in the operand ring");
  static_assert(8 * kXBufs * 8 <= 1024, "x barriers must fit in the epilogue's shared memory");
  extern __shared__ uint8_t smem_raw[];
  const gemm::Ctx c = gemm::setup<BN>(smem_raw, &map_a, &map_b);
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // the set-up above overlaps the previous kernel (the attention)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * gemm::kBM;
  const int kb_count = (p.K + gemm::kBK - 1) / gemm::kBK;

  if (warp == 0) {
    if (lane == 0) gemm::produce<BN>(c, &map_a, &map_b, m0, n0, kb_count, p.err, kErrGemmWait);
  } else if (warp == 1) {
    gemm::mma<BN>(c, kb_count, p.err, kErrGemmWait);
  } else if (warp >= 4) {
    // epilogue: warps 4-7 take rows 0-127 (accumulator columns [0, BN)),
    // warps 8-11 rows 128-255 ([BN, 2 BN)); a warp's 32 rows are its TMEM
    // lane quadrant, one row per lane.
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row_base = m0 + half * 128 + quad * 32;
    // while the MMAs run, pull this warp's 32 rows of x (BN columns) into L2
    {
      const int m = row_base + lane;
      const int ncols = min(BN, p.N - n0);
      if (m < p.M && ncols > 0) dev::prefetch_l2(p.x + static_cast<int64_t>(m) * p.N + n0, ncols * 4);
    }
    if (p.v_out == nullptr) {
      // x in 32 x 32 fp32 chunks staged by tensor-map loads in the idle
      // operand ring (128-byte swizzled, kXBufs in flight per warp); thread =
      // row: it adds dt * (v + bias) to its row of the chunk in place, taking
      // v straight from its TMEM lane, and a tensor-map store writes the
      // chunk back.  The loads hit L2 (x was prefetched during the MMAs).
      uint8_t* xb = c.smem + (warp - 4) * (kXBufs * kXChunkBytes);
      uint64_t* xbar = reinterpret_cast<uint64_t*>(c.smem + L::kExtra) + (warp - 4) * kXBufs;
      if (lane == 0) {
        dev::tma_prefetch_desc(&map_x);
        for (int i = 0; i < kXBufs; ++i) dev::mbar_init(&xbar[i], 1);
        dev::fence_barrier_init();
      }
      __syncwarp();
      const int nch = (min(BN, p.N - n0) + kXChunk - 1) / kXChunk;
      if (gemm::wait_acc(c, p.err, kErrGemmWait) && row_base < p.M) {
        if (lane == 0)
          for (int i = 0; i < kXBufs && i < nch; ++i) {
            dev::mbar_arrive_expect_tx(&xbar[i], kXChunkBytes);
            dev::tma_load_2d(xb + i * kXChunkBytes, &map_x, &xbar[i], n0 + i * kXChunk, row_base);
          }
        const uint32_t t_row = c.tmem + (static_cast<uint32_t>(quad * 32) << 16) + half * BN;
        const float dt = p.dt;
        #pragma unroll 1
        for (int cc = 0; cc < nch; ++cc) {
          const int bi = cc % kXBufs;
          uint32_t acc[32];
          dev::tmem_ld32(t_row + cc * kXChunk, acc);
          if (!__all_sync(0xffffffffu, dev::mbar_wait(&xbar[bi], (cc / kXBufs) & 1, c.abort))) {
            gemm::give_up(p.err, c.abort, kErrGemmWait, 4);
            break;
          }
          float4* row = reinterpret_cast<float4*>(xb + bi * kXChunkBytes + lane * 128);
          const int ncol0 = n0 + cc * kXChunk;
          #pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.bias && ncol0 + 4 * j < p.N) bb = *reinterpret_cast<const float4*>(p.bias + ncol0 + 4 * j);
            float4* cell = row + (j ^ (lane & 7));
            float4 y = *cell;
            y.x = fmaf(dt, __uint_as_float(acc[4 * j]) + bb.x, y.x);
            y.y = fmaf(dt, __uint_as_float(acc[4 * j + 1]) + bb.y, y.y);
            y.z = fmaf(dt, __uint_as_float(acc[4 * j + 2]) + bb.z, y.z);
            y.w = fmaf(dt, __uint_as_float(acc[4 * j + 3]) + bb.w, y.w);
            *cell = y;
          }
          dev::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            dev::tma_store_2d(&map_x, xb + bi * kXChunkBytes, ncol0, row_base);
            if (p.x_copy) dev::tma_store_2d(&map_xc, xb + bi * kXChunkBytes, ncol0, row_base);
            dev::bulk_commit();
            if (cc + kXBufs < nch) {
              // the buffer is reloaded once its store has read it
              dev::bulk_wait_read_all();
              dev::mbar_arrive_expect_tx(&xbar[bi], kXChunkBytes);
              dev::tma_load_2d(xb + bi * kXChunkBytes, &map_x, &xbar[bi], n0 + (cc + kXBufs) * kXChunk,
                               row_base);
            }
          }
        }
        if (lane == 0) dev::bulk_wait_all();
        __syncwarp();
      }
    } else if (gemm::wait_acc(c, p.err, kErrGemmWait)) {
      // with the velocity written out too (a debugging aid): each 32 x 32
      // chunk is turned around in shared memory and applied to x and v_out
      // with coalesced 128-byte row segments.  The operand ring is idle once
      // every MMA has completed: 4 KiB per warp
      float4* stage = reinterpret_cast<float4*>(c.smem + (warp - 4) * 4096);
      const uint32_t t_row = c.tmem + (static_cast<uint32_t>(quad * 32) << 16) + half * BN;
      const float dt = p.dt;
      const int seg = lane & 7;
      #pragma unroll 1
      for (int cc = 0; cc < BN; cc += 32) {
        uint32_t acc[32];
        dev::tmem_ld32(t_row + cc, acc);
        #pragma unroll
        for (int j = 0; j < 8; ++j)
          stage[lane * 8 + ((j + lane) & 7)] =
              make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                          __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
        __syncwarp();
        const int n = n0 + cc + 4 * seg;
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
    }
  }
  gemm::teardown<BN>(c);
}

// ------------------------------------------------------------ CTA-pair kernel
// Persistent CTA-pair GEMM (gemm_pair.cuh): a cluster of two CTAs computes
// 256 x 256 tiles of v with tcgen05.mma.cta_group::2, and each CTA keeps two
// 128 x 256 fp32 accumulators in TMEM, so the Euler epilogue of one tile (x
// through the shared-memory chunk staging above) runs while the next tile's
// MMAs accumulate into the other buffer, and the x read-modify-write traffic
// no longer idles the tensor cores.  Epilogue: warps 4-11, warp -> 32 rows
// (its TMEM lane quadrant) x 128 columns (one half of the tile).
namespace pair {
constexpr int kStages = 6;
using L = gemm_pair::Layout<kStages, 8>;  // one x barrier per epilogue warp
static_assert(kXChunkBytes == gemm_pair::kWarpStaging, "one x chunk per epilogue warp");
static_assert(L::kDynSmem <= 227 * 1024, "shared memory budget");
}  // namespace pair

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_pair::kThreads, 1)
    wo_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_xc,
                   const WoParams p, int n_tiles_n, int n_tiles) {
  using L = pair::L;
  extern __shared__ uint8_t smem_raw[];
  const gemm_pair::Ctx c = gemm_pair::setup<L>(smem_raw, &map_a, &map_b, &map_x);
  const gemm_pair::Hook hk{p.err, kErrGemmWait, p.fault_iter, p.wait_limit_ns};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kb_count = (p.K + gemm_pair::kBK - 1) / gemm_pair::kBK;
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // the set-up above overlaps the previous kernel (the attention)

  if (warp == 0) {
    if (lane == 0) gemm_pair::produce<L>(c, hk, &map_a, &map_b, n_tiles_n, n_tiles, kb_count);
  } else if (warp == 1) {
    if (c.leader) gemm_pair::mma<L>(c, hk, n_tiles, kb_count);
  } else if (warp == 2) {
    if (lane == 0 && !c.leader) gemm_pair::relay<L>(c, hk, n_tiles, kb_count);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;
    const int quad = warp & 3;
    const int ch = ew >> 2;
    uint8_t* xb = c.smem + L::kStaging + ew * kXChunkBytes;
    uint64_t* xbar = &c.bars[L::kExtraBar + ew];
    const uint32_t t_lane = c.tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float dt = p.dt;
    uint32_t xwaits = 0;
    int tile_i = 0;
    for (int t = c.cluster; t < n_tiles; t += c.n_clusters, ++tile_i) {
      const int buf = tile_i & 1;
      const int row_base = (t / n_tiles_n) * 256 + static_cast<int>(c.rank) * 128 + quad * 32;
      const int ncol0 = (t % n_tiles_n) * 256 + ch * 128;
      {
        // pull this warp's rows of x for the tile into L2 while the MMAs run
        const int m = row_base + lane;
        const int ncols = min(128, p.N - ncol0);
        if (m < p.M && ncols > 0) dev::prefetch_l2(p.x + static_cast<int64_t>(m) * p.N + ncol0, ncols * 4);
      }
      if (!gemm_pair::acc_wait<L>(c, hk, tile_i)) break;
      const int nch = row_base < p.M ? max(0, (min(128, p.N - ncol0) + kXChunk - 1) / kXChunk) : 0;
      if (lane == 0 && nch > 0) {
        dev::mbar_arrive_expect_tx(xbar, kXChunkBytes);
        dev::tma_load_2d(xb, &map_x, xbar, ncol0, row_base);
      }
      bool ok = true;
      #pragma unroll 1
      for (int cc = 0; cc < nch; ++cc) {
        uint32_t acc[32];
        dev::tmem_ld32(t_lane + static_cast<uint32_t>(buf * 256 + ch * 128 + cc * kXChunk), acc);
        const bool xg = __all_sync(0xffffffffu, dev::mbar_wait(xbar, xwaits & 1, c.abort, p.wait_limit_ns));
        ++xwaits;
        if (!xg) {
          gemm_pair::give_up(hk, c.abort, 16);
          ok = false;
          break;
        }
        float4* row = reinterpret_cast<float4*>(xb + lane * 128);
        const int n = ncol0 + cc * kXChunk;
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p.bias && n + 4 * j < p.N) bb = *reinterpret_cast<const float4*>(p.bias + n + 4 * j);
          float4* cell = row + (j ^ (lane & 7));
          float4 y = *cell;
          y.x = fmaf(dt, __uint_as_float(acc[4 * j]) + bb.x, y.x);
          y.y = fmaf(dt, __uint_as_float(acc[4 * j + 1]) + bb.y, y.y);
          y.z = fmaf(dt, __uint_as_float(acc[4 * j + 2]) + bb.z, y.z);
          y.w = fmaf(dt, __uint_as_float(acc[4 * j + 3]) + bb.w, y.w);
          *cell = y;
        }
        dev::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          dev::tma_store_2d(&map_x, xb, n, row_base);
          if (p.x_copy) dev::tma_store_2d(&map_xc, xb, n, row_base);
          dev::bulk_commit();
          if (cc + 1 < nch) {
            // the buffer is reloaded once its store has read it
            dev::bulk_wait_read_all();
            dev::mbar_arrive_expect_tx(xbar, kXChunkBytes);
            dev::tma_load_2d(xb, &map_x, xbar, n + kXChunk, row_base);
          }
        }
      }
      // this warp has read its part of the accumulator: release the buffer
      gemm_pair::acc_release<L>(c, tile_i);
      if (lane == 0) dev::bulk_wait_read_all();  // the staging buffer is reloaded by the next tile
      __syncwarp();
      if (!ok) break;
    }
    if (lane == 0) dev::bulk_wait_all();
    __syncwarp();
  }
  gemm_pair::teardown(c);
}

template <int BN>
int launch_bn(const void* o, const void* w, const float* bias, float* x, int64_t M, int K, int N,
              float dt, float* v_out, float* x_copy, cudaStream_t stream) {
  using L = gemm::Layout<BN>;
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
  const uint32_t ba[2] = {gemm::kBK, 128};
  int rc = encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N};
  const uint32_t bb[2] = {gemm::kBK, BN};
  rc = encode_tiled(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, db, sa, bb, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  CUtensorMap mx, mxc;
  const uint64_t dx[2] = {(uint64_t)N, (uint64_t)M};
  const uint64_t sx[1] = {(uint64_t)N * 4};
  const uint32_t bx[2] = {kXChunk, 32};
  rc = encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, x, dx, sx, bx, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  rc = encode_tiled(&mxc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, x_copy ? x_copy : x, dx, sx, bx,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  WoParams p{(int)M, N, K, dt, bias, x, v_out, nullptr, -1, dev::kWaitLimitNs, x_copy};
  if ((rc = error_word(&p.err))) return rc;
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + gemm::kBM - 1) / gemm::kBM));
  SAVGB_CUDA(launch_dependent(wo_euler_kernel<BN>, grid, dim3(gemm::kThreads), L::kDynSmem, stream, ma, mb, mx,
                              mxc, p));
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

}  // namespace

int validate_out_proj(const void* o, const void* w, const float* bias, const float* x, int64_t M,
                      int hid_in, int hid_out, const float* v_out) {
  if (!o || !w || !x) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: null o, w_o or x");
  if (!aligned16(o) || !aligned16(w) || !aligned16(x) || (bias && !aligned16(bias)) ||
      (v_out && !aligned16(v_out)))
    return fail(SAVGB_ERR_ALIGNMENT, "out_proj_euler_step: pointers must be 16-byte aligned");
  if (M < 1 || M > ((int64_t)1 << 31) - 1 - gemm::kBM) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: M must be in [1, 2^31)");
  if (hid_in < 8 || hid_in % 8) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hid_in must be a positive multiple of 8");
  if (hid_out < 16 || hid_out % 16) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hid_out must be a positive multiple of 16");
  if (hid_in > (1 << 24) || hid_out > (1 << 24)) return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler_step: hidden size too large");
  return SAVGB_OK;
}

// The persistent CTA-pair kernel: x updated alone (no velocity output), the
// output width a multiple of 256.
int launch_pair(const void* o, const void* w, const float* bias, float* x, int64_t M, int K, int N, float dt,
                float* x_copy, int sms, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  static int max_clusters[64] = {0};
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (!attr_done[dev_id & 63]) {
    SAVGB_CUDA(cudaFuncSetAttribute(wo_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    pair::L::kDynSmem));
    int rc = gemm_pair::max_clusters(wo_pair_kernel, sms, pair::L::kDynSmem, &max_clusters[dev_id & 63]);
    if (rc) return rc;
    attr_done[dev_id & 63] = true;
  }
  CUtensorMap ma, mb, mx, mxc;
  const uint64_t da[2] = {(uint64_t)K, (uint64_t)M};
  const uint64_t sa[1] = {(uint64_t)K * 2};
  const uint32_t box128[2] = {gemm_pair::kBK, 128};
  int rc = encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o, da, sa, box128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t db[2] = {(uint64_t)K, (uint64_t)N};
  rc = encode_tiled(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, db, sa, box128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t dx[2] = {(uint64_t)N, (uint64_t)M};
  const uint64_t sx[1] = {(uint64_t)N * 4};
  const uint32_t bx[2] = {kXChunk, 32};
  rc = encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, x, dx, sx, bx, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  rc = encode_tiled(&mxc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, x_copy ? x_copy : x, dx, sx, bx,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  WoParams p{(int)M, N, K, dt, bias, x, nullptr, nullptr, -1, dev::kWaitLimitNs, x_copy};
  if ((rc = error_word(&p.err))) return rc;
  ArmedFault fault;
  if (take_fault(SAVGB_FAULT_WO_PAIR_RELAY, &fault)) {
    p.fault_iter = fault.index;
    p.wait_limit_ns = fault.limit_ns;
  }
  const int n_tiles_n = N / 256;
  const int n_tiles = (int)((M + 255) / 256) * n_tiles_n;
  // one wave of pairs: as many clusters as can be resident at once
  const int clusters = std::min(n_tiles, max_clusters[dev_id & 63]);
  SAVGB_CUDA(launch_dependent(wo_pair_kernel, dim3((unsigned)(2 * clusters)), dim3(gemm_pair::kThreads),
                              pair::L::kDynSmem, stream, ma, mb, mx, mxc, p, n_tiles_n, n_tiles));
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

int launch_out_proj_euler(const void* o, const void* w, const float* bias, float* x, int64_t M,
                          int hid_in, int hid_out, float dt, float* v_out, cudaStream_t stream, float* x_copy) {
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  if (x_copy && (v_out || !aligned16(x_copy)))
    return fail(SAVGB_ERR_INVALID_ARG, "out_proj_euler: a copy of x needs no v_out and a 16-byte aligned buffer");
  if (v_out == nullptr && hid_out % 256 == 0)
    return launch_pair(o, w, bias, x, M, hid_in, hid_out, dt, x_copy, sms, stream);
  if (hid_out % 256 == 0)
    return launch_bn<256>(o, w, bias, x, M, hid_in, hid_out, dt, v_out, x_copy, stream);
  return launch_bn<128>(o, w, bias, x, M, hid_in, hid_out, dt, v_out, x_copy, stream);
}

}  // namespace savgb

extern "C" int out_proj_euler_step(const void* o, const void* w_o, const float* bias, float* x,
                                   int64_t M, int hid_in, int hid_out, float dt, float* v_out,
                                   void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:out_proj_euler_step");
  clear_error();
  int rc = validate_out_proj(o, w_o, bias, x, M, hid_in, hid_out, v_out);
  if (rc) return rc;
  return launch_out_proj_euler(o, w_o, bias, x, M, hid_in, hid_out, dt, v_out,
                               static_cast<cudaStream_t>(stream));
}
