// QKV projection of one DiT attention block, with the 3D RoPE of q and k in
// the GEMM epilogue, and the fp32 -> bf16 conversion of its input.
//
//   [q | k | v] = x W_qkv^T,  W_qkv = [W_q; W_k; W_v]  (bf16 [3*hid][hid])
//   q, k rotated at their chunk-local (t, h, w) positions; v as is.
//
// HeyGen, "Avatar inference at scale", section "The underlying model
// architecture": the denoiser is a Diffusion Transformer; one attention block
// with stand-in weights (its own QKV and output projections) takes the place
// of the whole network in this library.  The rotation follows rope3d_apply's
// reading (D/2 pairs split [t | h | w], pair j of an axis with P pairs
// turning at base^(-j/P)).
//
// Two kernels share one epilogue.  When 3*H*D is a multiple of 256 and the
// cos/sin tables fit next to its ring, a persistent CTA-pair GEMM
// (gemm_pair.cuh) computes 256 x 256 tiles with double-buffered accumulators,
// so each tile's epilogue overlaps the MMAs of the cluster's next tile;
// otherwise one CTA computes one 256 x BN tile (gemm_tc.cuh).  The epilogue
// warps build the cos/sin tables of the three axes in shared memory while the
// MMAs run; then each 32-column chunk of an accumulator row (one head's
// channels) is rotated pair by pair if it belongs to q or k, rounded to bf16,
// turned around in shared memory and stored with coalesced 64-byte row
// segments.  With a tail buffer, the unrotated k of the last n_tail tokens of
// every batch is also stored there (the next chunk's boundary before its
// RoPE).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "common.h"
#include "gemm_pair.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace savgb {
namespace {

struct QkvParams {
  int M, N3, K;  // rows (B * n_tok), 3 * hid, hid
  int hid, D, n_tok;
  int gt, gh, gw, t0;
  int p_t, p_h, p_w;
  float log2_base;
  __nv_bfloat16* q;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  __nv_bfloat16* k_tail;  // optional, [B][n_tail][hid]
  int n_tail;
  DeviceErrorWord* err;
};

// Cos/sin tables [t | h | w] x pairs of each axis in shared memory, built by
// the 256 epilogue threads (threadIdx.x 128..383), then a barrier among them.
__device__ __forceinline__ void build_tables(float2* tab, const QkvParams& p) {
  const int n_t = p.gt * p.p_t, n_h = p.gh * p.p_h, n_w = p.gw * p.p_w;
  for (int i = threadIdx.x - 128; i < n_t + n_h + n_w; i += 256) {
    int pos, j, P;
    if (i < n_t) { pos = p.t0 + i / p.p_t; j = i % p.p_t; P = p.p_t; }
    else if (i < n_t + n_h) { const int kk = i - n_t; pos = kk / p.p_h; j = kk % p.p_h; P = p.p_h; }
    else { const int kk = i - n_t - n_h; pos = kk / p.p_w; j = kk % p.p_w; P = p.p_w; }
    const float omega = exp2f(-static_cast<float>(j) / static_cast<float>(P) * p.log2_base);
    float sn, cs;
    sincosf(static_cast<float>(pos) * omega, &sn, &cs);
    tab[i] = make_float2(cs, sn);
  }
  dev::named_barrier_256();  // the eight epilogue warps (no waits before it)
}

// One accumulator row of an epilogue thread: its token and table rows.
struct QkvRow {
  int b, tk;
  const float2 *tr, *hr, *wr;
  bool tail;
};

__device__ __forceinline__ QkvRow qkv_row(const float2* tab, const QkvParams& p, int m) {
  QkvRow r;
  r.b = m / p.n_tok;
  r.tk = m - r.b * p.n_tok;
  const int hw = p.gh * p.gw;
  const int tt = r.tk / hw;
  const int r2 = r.tk - tt * hw;
  const int hh = r2 / p.gw;
  const int ww = r2 - hh * p.gw;
  const int n_t = p.gt * p.p_t, n_h = p.gh * p.p_h;
  r.tr = tab + tt * p.p_t;
  r.hr = tab + n_t + hh * p.p_h - p.p_t;
  r.wr = tab + n_t + n_h + ww * p.p_w - p.p_t - p.p_h;
  r.tail = p.k_tail != nullptr && m < p.M && r.tk >= p.n_tok - p.n_tail;
  return r;
}

// One 32 x 32 chunk of a warp (its 32 rows from row_base, columns n ..
// n+31 of [q | k | v], one head's channels): rotate q and k pairs, round to
// bf16, store the unrotated k of tail rows, turn the chunk around in `stage`
// (4 KiB) and write it with coalesced 64-byte row segments.
__device__ __forceinline__ void qkv_store_chunk(const QkvParams& p, const QkvRow& r, const uint32_t (&acc)[32], int n,
                                                int row_base, uint4* stage) {
  const int lane = threadIdx.x & 31;
  const int section = n / p.hid;  // 0 q, 1 k, 2 v (a 32-column chunk lies in one)
  const int nn = n - section * p.hid;
  const int pair0 = (nn % p.D) >> 1;
  const int ph_end = p.p_t + p.p_h;
  uint32_t raw[16], out[16];
  #pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float a = __uint_as_float(acc[2 * i]), bb = __uint_as_float(acc[2 * i + 1]);
    raw[i] = dev::pack_bf16x2(a, bb);
    if (section < 2) {
      const int pr = pair0 + i;
      const float2 cs = pr < p.p_t ? r.tr[pr] : (pr < ph_end ? r.hr[pr] : r.wr[pr]);
      out[i] = dev::pack_bf16x2(a * cs.x - bb * cs.y, a * cs.y + bb * cs.x);
    } else {
      out[i] = raw[i];
    }
  }
  if (section == 1 && r.tail) {
    uint4* dst = reinterpret_cast<uint4*>(
        p.k_tail + (static_cast<int64_t>(r.b) * p.n_tail + r.tk - (p.n_tok - p.n_tail)) * p.hid + nn);
    #pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(raw[4 * i], raw[4 * i + 1], raw[4 * i + 2], raw[4 * i + 3]);
  }
  // turn the 32 x 32 bf16 chunk around: row r's 64 bytes, 4 x 16 B, rotated by r
  #pragma unroll
  for (int j = 0; j < 4; ++j)
    stage[lane * 4 + ((j + lane) & 3)] = make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
  __syncwarp();
  __nv_bfloat16* base = section == 0 ? p.q : (section == 1 ? p.k : p.v);
  const int qd = lane & 3;
  #pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const int rr = 8 * kk + (lane >> 2);
    const int mr = row_base + rr;
    if (mr < p.M)
      *reinterpret_cast<uint4*>(base + static_cast<int64_t>(mr) * p.hid + nn + 8 * qd) =
          stage[rr * 4 + ((qd + rr) & 3)];
  }
  __syncwarp();
}

template <int BN>
__global__ void __launch_bounds__(gemm::kThreads, 1)
    qkv_rope_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const QkvParams p) {
  using L = gemm::Layout<BN>;
  extern __shared__ uint8_t smem_raw[];
  const gemm::Ctx c = gemm::setup<BN>(smem_raw, &map_a, &map_b);
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
    // cos/sin tables, built while the MMAs run
    float2* tab = reinterpret_cast<float2*>(c.smem + L::kExtra);
    build_tables(tab, p);
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row_base = m0 + half * 128 + quad * 32;
    const QkvRow r = qkv_row(tab, p, row_base + lane);
    if (gemm::wait_acc(c, p.err, kErrGemmWait)) {
      uint4* stage = reinterpret_cast<uint4*>(c.smem + (warp - 4) * 4096);
      const uint32_t t_row = c.tmem + (static_cast<uint32_t>(quad * 32) << 16) + half * BN;
      #pragma unroll 1
      for (int cc = 0; cc < BN; cc += 32) {
        const int n = n0 + cc;
        if (n >= p.N3) break;  // uniform: the tile's last columns lie past 3*hid
        uint32_t acc[32];
        dev::tmem_ld32(t_row + cc, acc);
        qkv_store_chunk(p, r, acc, n, row_base, stage);
      }
    }
  }
  gemm::teardown<BN>(c);
}

// ------------------------------------------------------------ CTA-pair kernel
namespace qpair {
constexpr int kStages = 5;  // leaves room for the cos/sin tables after the ring
using L = gemm_pair::Layout<kStages, 0>;
}  // namespace qpair

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_pair::kThreads, 1)
    qkv_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const QkvParams p, int n_tiles_n, int n_tiles) {
  using L = qpair::L;
  extern __shared__ uint8_t smem_raw[];
  const gemm_pair::Ctx c = gemm_pair::setup<L>(smem_raw, &map_a, &map_b, nullptr);
  const gemm_pair::Hook hk{p.err, kErrGemmWait, -1, dev::kWaitLimitNs};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kb_count = (p.K + gemm_pair::kBK - 1) / gemm_pair::kBK;
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // the set-up above overlaps the previous kernel (the bf16 copy of x)

  if (warp == 0) {
    if (lane == 0) gemm_pair::produce<L>(c, hk, &map_a, &map_b, n_tiles_n, n_tiles, kb_count);
  } else if (warp == 1) {
    if (c.leader) gemm_pair::mma<L>(c, hk, n_tiles, kb_count);
  } else if (warp == 2) {
    if (lane == 0 && !c.leader) gemm_pair::relay<L>(c, hk, n_tiles, kb_count);
  } else if (warp >= 4) {
    float2* tab = reinterpret_cast<float2*>(c.smem + L::kExtra);
    build_tables(tab, p);
    const int ew = warp - 4;
    const int quad = warp & 3;
    const int ch = ew >> 2;  // which 128-column half of the tile
    uint4* stage = reinterpret_cast<uint4*>(c.smem + L::kStaging + ew * gemm_pair::kWarpStaging);
    const uint32_t t_lane = c.tmem + (static_cast<uint32_t>(quad * 32) << 16);
    int tile_i = 0;
    for (int t = c.cluster; t < n_tiles; t += c.n_clusters, ++tile_i) {
      const int buf = tile_i & 1;
      const int row_base = (t / n_tiles_n) * 256 + static_cast<int>(c.rank) * 128 + quad * 32;
      const int ncol0 = (t % n_tiles_n) * 256 + ch * 128;
      const QkvRow r = qkv_row(tab, p, row_base + lane);
      if (!gemm_pair::acc_wait<L>(c, hk, tile_i)) break;
      if (row_base < p.M) {
        #pragma unroll 1
        for (int cc = 0; cc < 128; cc += 32) {
          uint32_t acc[32];
          dev::tmem_ld32(t_lane + static_cast<uint32_t>(buf * 256 + ch * 128 + cc), acc);
          qkv_store_chunk(p, r, acc, ncol0 + cc, row_base, stage);
        }
      }
      // this warp has read its part of the accumulator: release the buffer
      gemm_pair::acc_release<L>(c, tile_i);
    }
  }
  gemm_pair::teardown(c);
}

// fp32 -> bf16 (round to nearest even), 8 elements per thread per iteration.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float4* __restrict__ x, uint4* __restrict__ y,
                                                      int64_t n8) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(x + 2 * i);
    const float4 b = __ldcs(x + 2 * i + 1);
    __stcs(y + i, make_uint4(dev::pack_bf16x2(a.x, a.y), dev::pack_bf16x2(a.z, a.w), dev::pack_bf16x2(b.x, b.y),
                             dev::pack_bf16x2(b.z, b.w)));
  }
}

QkvParams qkv_params(const QkvArgs& a) {
  QkvParams p{};
  const int hid = a.H * a.D;
  p.M = (int)(a.B * a.n_tokens);
  p.N3 = 3 * hid;
  p.K = hid;
  p.hid = hid;
  p.D = a.D;
  p.n_tok = (int)a.n_tokens;
  p.gt = a.grid_t; p.gh = a.grid_h; p.gw = a.grid_w; p.t0 = a.t0;
  const int P = a.D / 2;
  p.p_h = P / 3;
  p.p_w = P / 3;
  p.p_t = P - 2 * (P / 3);
  p.log2_base = (float)std::log2(a.base);
  p.q = static_cast<__nv_bfloat16*>(a.q);
  p.k = static_cast<__nv_bfloat16*>(a.k);
  p.v = static_cast<__nv_bfloat16*>(a.v);
  p.k_tail = static_cast<__nv_bfloat16*>(a.k_tail);
  p.n_tail = (int)a.n_tail;
  return p;
}

// Bytes of the cos/sin tables of the three axes.
int64_t qkv_table_bytes(const QkvParams& p) {
  return 8 * ((int64_t)p.gt * p.p_t + (int64_t)p.gh * p.p_h + (int64_t)p.gw * p.p_w);
}

int qkv_maps(const QkvArgs& a, const QkvParams& p, uint32_t b_rows, CUtensorMap* ma, CUtensorMap* mb) {
  const uint64_t da[2] = {(uint64_t)p.hid, (uint64_t)p.M};
  const uint64_t sa[1] = {(uint64_t)p.hid * 2};
  const uint32_t ba[2] = {gemm::kBK, 128};
  int rc = encode_tiled(ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x_bf16, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t db[2] = {(uint64_t)p.hid, (uint64_t)p.N3};
  const uint32_t bb[2] = {gemm::kBK, b_rows};
  return encode_tiled(mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w_qkv, db, sa, bb, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int BN>
int launch_qkv_bn(const QkvArgs& a, cudaStream_t stream) {
  using L = gemm::Layout<BN>;
  static bool attr_done[64] = {false};
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (!attr_done[dev_id & 63]) {
    SAVGB_CUDA(cudaFuncSetAttribute(qkv_rope_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
    attr_done[dev_id & 63] = true;
  }
  QkvParams p = qkv_params(a);
  int rc = error_word(&p.err);
  if (rc) return rc;
  const int64_t tab = qkv_table_bytes(p);
  if (L::kDynSmem + tab > 227 * 1024)
    return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: RoPE tables of %lld bytes do not fit", (long long)tab);
  CUtensorMap ma, mb;
  if ((rc = qkv_maps(a, p, BN, &ma, &mb))) return rc;
  dim3 grid((unsigned)((p.N3 + BN - 1) / BN), (unsigned)((p.M + gemm::kBM - 1) / gemm::kBM));
  qkv_rope_kernel<BN><<<grid, gemm::kThreads, (int)(L::kDynSmem + tab), stream>>>(ma, mb, p);
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

// The persistent CTA-pair kernel: 3*hid a multiple of 256 and the tables
// fitting after its ring (checked by the caller).
int launch_qkv_pair(const QkvArgs& a, int sms, cudaStream_t stream) {
  using L = qpair::L;
  QkvParams p = qkv_params(a);
  int rc = error_word(&p.err);
  if (rc) return rc;
  const int smem = L::kDynSmem + (int)qkv_table_bytes(p);
  static int attr_smem[64] = {0};
  static int max_clusters[64] = {0};
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (attr_smem[dev_id & 63] == 0) {
    SAVGB_CUDA(cudaFuncSetAttribute(qkv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
    attr_smem[dev_id & 63] = 1;
  }
  if (max_clusters[dev_id & 63] == 0 &&
      (rc = gemm_pair::max_clusters(qkv_pair_kernel, sms, 227 * 1024, &max_clusters[dev_id & 63])))
    return rc;
  CUtensorMap ma, mb;
  if ((rc = qkv_maps(a, p, 128, &ma, &mb))) return rc;
  const int n_tiles_n = p.N3 / 256;
  const int n_tiles = ((p.M + 255) / 256) * n_tiles_n;
  const int clusters = std::min(n_tiles, max_clusters[dev_id & 63]);
  SAVGB_CUDA(launch_dependent(qkv_pair_kernel, dim3((unsigned)(2 * clusters)), dim3(gemm_pair::kThreads), smem,
                              stream, ma, mb, p, n_tiles_n, n_tiles));
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

bool qkv_pair_fits(const QkvArgs& a) {
  const QkvParams p = qkv_params(a);
  return p.N3 % 256 == 0 && qpair::L::kDynSmem + qkv_table_bytes(p) <= 227 * 1024;
}

}  // namespace

int validate_qkv(const QkvArgs& a) {
  if (!a.x_bf16 || !a.w_qkv || !a.q || !a.k || !a.v) return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: null pointer");
  if (!aligned16(a.x_bf16) || !aligned16(a.w_qkv) || !aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) ||
      (a.k_tail && !aligned16(a.k_tail)))
    return fail(SAVGB_ERR_ALIGNMENT, "qkv_rope_project: pointers must be 16-byte aligned");
  if (a.D != 64 && a.D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "qkv_rope_project: head_dim %d (64 or 128)", a.D);
  if (a.B < 1 || a.H < 1 || a.n_tokens < 1) return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: B, H, n_tokens >= 1");
  if ((int64_t)a.grid_t * a.grid_h * a.grid_w != a.n_tokens)
    return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: n_tokens != grid_t*grid_h*grid_w");
  if (a.grid_t > 4096 || a.grid_h > 4096 || a.grid_w > 4096)
    return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: grid sizes must be <= 4096");
  if (!(a.base > 0.0) || !std::isfinite(a.base)) return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: base must be > 0");
  if ((double)a.B * a.n_tokens > 2147483647.0 - 256) return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: too many rows");
  if (a.k_tail && (a.n_tail < 1 || a.n_tail > a.n_tokens))
    return fail(SAVGB_ERR_INVALID_ARG, "qkv_rope_project: n_tail must be in [1, n_tokens]");
  return SAVGB_OK;
}

int launch_qkv_rope(const QkvArgs& a, cudaStream_t stream) {
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  if (qkv_pair_fits(a)) return launch_qkv_pair(a, sms, stream);
  if ((3 * a.H * a.D) % 256 == 0) return launch_qkv_bn<256>(a, stream);
  return launch_qkv_bn<128>(a, stream);
}

int launch_to_bf16(const float* x, void* y, int64_t n, cudaStream_t stream) {
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  if (n % 8 || !aligned16(x) || !aligned16(y)) return fail(SAVGB_ERR_ALIGNMENT, "to_bf16: n % 8 and 16-byte pointers");
  const int64_t n8 = n / 8;
  int64_t blocks = (n8 + 255) / 256;
  if (blocks > 8 * sms) blocks = 8 * sms;
  to_bf16_kernel<<<(unsigned)(blocks > 0 ? blocks : 1), 256, 0, stream>>>(reinterpret_cast<const float4*>(x),
                                                                           static_cast<uint4*>(y), n8);
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

}  // namespace savgb

extern "C" int qkv_rope_project(const void* x_bf16, const void* w_qkv, void* q, void* k, void* v, int B,
                                int64_t n_tokens, int H, int D, int grid_t, int grid_h, int grid_w, int t0,
                                double base, void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:qkv_rope_project");
  clear_error();
  QkvArgs a{x_bf16, w_qkv, q, k, v, nullptr, 0, B, n_tokens, H, D, grid_t, grid_h, grid_w, t0, base};
  int rc = validate_qkv(a);
  if (rc) return rc;
  return launch_qkv_rope(a, static_cast<cudaStream_t>(stream));
}
