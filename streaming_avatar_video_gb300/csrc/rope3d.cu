// 3D (t, h, w) rotary position embedding of bf16 token tensors.
//
// Positions of the chunked latent video (HeyGen, "Avatar inference at scale",
// section "The underlying model architecture").  The D/2 channel pairs are
// split [t | h | w] (spatial axes floor(D/6) pairs each, time the rest); pair
// j of an axis with P pairs turns at base^(-j/P) radians per position.
//
// HBM-bound: each element is read once and written once.  Each block first
// builds the cos/sin tables of the three axes in shared memory (fp32, from
// sincosf); then a warp takes one token at a time, decodes its (t, h, w)
// once and streams its 16-byte vectors (8 channels = 4 pairs of one head),
// eight per lane in flight.
#include <cuda_bf16.h>

#include <cmath>

#include "common.h"
#include "ptx.cuh"

namespace savgb {
namespace {

constexpr int kRopeThreads = 256;  // 8 warps; a warp rotates one token at a time
constexpr int kRopeWarps = kRopeThreads / 32;
constexpr int kRopeBatch = 8;      // 16-byte vectors of a token in flight per lane
constexpr int kRopeMaxTableBytes = 96 * 1024;

struct RopeTensor {
  const uint4* in;
  uint4* out;
  int64_t in_bs;   // 16-byte vectors between batches
  int64_t out_bs;
};

struct RopeKernelArgs {
  RopeTensor t[2];
  int n_tokens, vec_per_tok, vec_per_head;  // vec_per_head = D/8
  int gh, gw, gt, t0;
  int p_t, p_h, p_w;
  float log2_base;
};

__device__ __forceinline__ void rotate_pair(uint32_t& packed, float2 cs) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&packed);
  const float a = __low2float(v);
  const float b = __high2float(v);
  const float ra = a * cs.x - b * cs.y;
  const float rb = a * cs.y + b * cs.x;
  __nv_bfloat162 r = __floats2bfloat162_rn(ra, rb);
  packed = *reinterpret_cast<uint32_t*>(&r);
}

// Builds the block's cos/sin tables of the three axes in shared memory.
__device__ __forceinline__ void build_tables(float2* tab, const RopeKernelArgs& a) {
  const int n_t = a.gt * a.p_t, n_h = a.gh * a.p_h, n_w = a.gw * a.p_w;
  for (int i = threadIdx.x; i < n_t + n_h + n_w; i += blockDim.x) {
    int pos, j, P;
    if (i < n_t) {
      pos = a.t0 + i / a.p_t; j = i % a.p_t; P = a.p_t;
    } else if (i < n_t + n_h) {
      const int k = i - n_t; pos = k / a.p_h; j = k % a.p_h; P = a.p_h;
    } else {
      const int k = i - n_t - n_h; pos = k / a.p_w; j = k % a.p_w; P = a.p_w;
    }
    const float omega = exp2f(-static_cast<float>(j) / static_cast<float>(P) * a.log2_base);
    float s, c;
    sincosf(static_cast<float>(pos) * omega, &s, &c);
    tab[i] = make_float2(c, s);
  }
}

// grid: (token groups, B, tensors).  Each block builds the cos/sin tables of
// the three axes in shared memory, then each warp takes whole tokens: the
// token's (t, h, w) is decoded once and its H*D/8 vectors are streamed with
// kRopeBatch loads in flight per lane.  General shapes.
__global__ void __launch_bounds__(kRopeThreads) rope3d_kernel(const RopeKernelArgs a) {
  extern __shared__ float2 tab[];
  float2* tab_t = tab;
  float2* tab_h = tab_t + a.gt * a.p_t;
  float2* tab_w = tab_h + a.gh * a.p_h;
  dev::griddep_launch_dependents();
  build_tables(tab, a);
  __syncthreads();
  dev::griddep_wait();

  const int ti = blockIdx.z;
  const int b = blockIdx.y;
  const uint4* __restrict__ in = (ti == 0 ? a.t[0].in : a.t[1].in) + b * (ti == 0 ? a.t[0].in_bs : a.t[1].in_bs);
  uint4* __restrict__ out = (ti == 0 ? a.t[0].out : a.t[1].out) + b * (ti == 0 ? a.t[0].out_bs : a.t[1].out_bs);
  const int lane = threadIdx.x & 31;
  const int hw = a.gh * a.gw;
  const int vpt = a.vec_per_tok;
  const int ph_end = a.p_t + a.p_h;
  for (int n = blockIdx.x * kRopeWarps + (threadIdx.x >> 5); n < a.n_tokens; n += gridDim.x * kRopeWarps) {
    const int tt = n / hw;
    const int r2 = n - tt * hw;
    const int hh = r2 / a.gw;
    const int ww = r2 - hh * a.gw;
    const float2* tr = tab_t + tt * a.p_t;
    const float2* hr = tab_h + hh * a.p_h - a.p_t;
    const float2* wr = tab_w + ww * a.p_w - ph_end;
    const uint4* src = in + static_cast<int64_t>(n) * vpt;
    uint4* dst = out + static_cast<int64_t>(n) * vpt;
    for (int j0 = 0; j0 < vpt; j0 += 32 * kRopeBatch) {
      uint4 v[kRopeBatch];
      #pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int j = j0 + lane + 32 * u;
        if (j < vpt) v[u] = __ldcs(src + j);
      }
      #pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int j = j0 + lane + 32 * u;
        if (j < vpt) {
          const int p0 = (j % a.vec_per_head) * 4;
          uint32_t w0 = v[u].x, w1 = v[u].y, w2 = v[u].z, w3 = v[u].w;
          #define SAVGB_ROT(W, Q) { const int p_ = p0 + (Q); \
            const float2 cs_ = p_ < a.p_t ? tr[p_] : (p_ < ph_end ? hr[p_] : wr[p_]); \
            rotate_pair(W, cs_); }
          SAVGB_ROT(w0, 0) SAVGB_ROT(w1, 1) SAVGB_ROT(w2, 2) SAVGB_ROT(w3, 3)
          #undef SAVGB_ROT
          __stcs(dst + j, make_uint4(w0, w1, w2, w3));
        }
      }
    }
  }
}

// Shapes whose token holds a whole number of warp-widths of 16-byte vectors
// (vec_per_tok = 32*upl, upl <= kRopeFastMax) and whose head holds a divisor
// of 32 vectors: lane L then always meets the same four channel pairs
// ((L mod D/8)*4 ...), so it looks its four (cos, sin) up once per token and
// applies them to all upl of its vectors.  The tables are built before the
// wait on the previous kernel of the stream, so they overlap its tail.
constexpr int kRopeFastMax = 12;

__global__ void __launch_bounds__(kRopeThreads) rope3d_fast_kernel(const RopeKernelArgs a) {
  extern __shared__ float2 tab[];
  const int ti = blockIdx.z;
  const int b = blockIdx.y;
  const uint4* __restrict__ in = (ti == 0 ? a.t[0].in : a.t[1].in) + b * (ti == 0 ? a.t[0].in_bs : a.t[1].in_bs);
  uint4* __restrict__ out = (ti == 0 ? a.t[0].out : a.t[1].out) + b * (ti == 0 ? a.t[0].out_bs : a.t[1].out_bs);
  const int lane = threadIdx.x & 31;
  const int vpt = a.vec_per_tok;
  const int upl = vpt >> 5;
  const int stride = gridDim.x * kRopeWarps;
  int n = blockIdx.x * kRopeWarps + (threadIdx.x >> 5);
  uint4 v[kRopeFastMax];
  auto load = [&](int tok) {
    const uint4* src = in + static_cast<int64_t>(tok) * vpt + lane;
    #pragma unroll
    for (int u = 0; u < kRopeFastMax; ++u)
      if (u < upl) v[u] = __ldcs(src + 32 * u);
  };
  dev::griddep_launch_dependents();
  build_tables(tab, a);
  dev::griddep_wait();
  if (n < a.n_tokens) load(n);
  __syncthreads();

  const float2* tab_t = tab;
  const float2* tab_h = tab_t + a.gt * a.p_t;
  const float2* tab_w = tab_h + a.gh * a.p_h;
  const int hw = a.gh * a.gw;
  const int ph_end = a.p_t + a.p_h;
  const int p0 = (lane % a.vec_per_head) * 4;
  for (; n < a.n_tokens; n += stride) {
    const int tt = n / hw;
    const int r2 = n - tt * hw;
    const int hh = r2 / a.gw;
    const int ww = r2 - hh * a.gw;
    float2 cs[4];
    #pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int p_ = p0 + q;
      cs[q] = p_ < a.p_t ? tab_t[tt * a.p_t + p_]
                         : (p_ < ph_end ? tab_h[hh * a.p_h + p_ - a.p_t] : tab_w[ww * a.p_w + p_ - ph_end]);
    }
    uint4* dst = out + static_cast<int64_t>(n) * vpt + lane;
    #pragma unroll
    for (int u = 0; u < kRopeFastMax; ++u) {
      if (u < upl) {
        uint32_t w0 = v[u].x, w1 = v[u].y, w2 = v[u].z, w3 = v[u].w;
        rotate_pair(w0, cs[0]);
        rotate_pair(w1, cs[1]);
        rotate_pair(w2, cs[2]);
        rotate_pair(w3, cs[3]);
        __stcs(dst + 32 * u, make_uint4(w0, w1, w2, w3));
      }
    }
    if (n + stride < a.n_tokens) load(n + stride);
  }
}

void axis_split(int D, int* pt, int* ph, int* pw) {
  const int P = D / 2;
  *ph = P / 3;
  *pw = P / 3;
  *pt = P - 2 * (P / 3);
}

size_t table_bytes(const RopeArgs& a) {
  int pt, ph, pw;
  axis_split(a.D, &pt, &ph, &pw);
  return sizeof(float2) * ((size_t)a.grid_t * pt + (size_t)a.grid_h * ph + (size_t)a.grid_w * pw);
}

}  // namespace

int validate_rope(const RopeArgs& a) {
  if (!a.in || !a.out) return fail(SAVGB_ERR_INVALID_ARG, "rope3d: null pointer");
  if (!aligned16(a.in) || !aligned16(a.out)) return fail(SAVGB_ERR_ALIGNMENT, "rope3d: pointers must be 16-byte aligned");
  if (a.B < 1 || a.B > 65535 || a.H < 1 || a.n_tokens < 1) return fail(SAVGB_ERR_INVALID_ARG, "rope3d: B must be in [1, 65535], H and n_tokens >= 1");
  if (a.D < 8 || a.D > 256 || a.D % 8) return fail(SAVGB_ERR_INVALID_ARG, "rope3d: D must be a multiple of 8 in [8, 256]");
  if (a.grid_t < 1 || a.grid_h < 1 || a.grid_w < 1 || a.grid_t > 4096 || a.grid_h > 4096 ||
      a.grid_w > 4096)
    return fail(SAVGB_ERR_INVALID_ARG, "rope3d: grid sizes must be in [1, 4096]");
  if ((int64_t)a.grid_t * a.grid_h * a.grid_w != a.n_tokens)
    return fail(SAVGB_ERR_INVALID_ARG, "rope3d: n_tokens (%lld) != grid_t*grid_h*grid_w (%lld)",
                (long long)a.n_tokens, (long long)a.grid_t * a.grid_h * a.grid_w);
  if (!(a.base > 0.0) || !std::isfinite(a.base)) return fail(SAVGB_ERR_INVALID_ARG, "rope3d: base must be finite and > 0");
  if (a.t0 < -(1 << 20) || a.t0 > (1 << 20)) return fail(SAVGB_ERR_INVALID_ARG, "rope3d: |t0| > 2^20");
  if ((double)a.B * a.n_tokens * a.H * (a.D / 8) >= 2147483647.0)
    return fail(SAVGB_ERR_INVALID_ARG, "rope3d: more than 2^31 16-byte vectors");
  if (table_bytes(a) > (size_t)kRopeMaxTableBytes)
    return fail(SAVGB_ERR_INVALID_ARG, "rope3d: angle tables need %zu bytes (> %d)", table_bytes(a), kRopeMaxTableBytes);
  return SAVGB_OK;
}

static int launch_rope_multi(const RopeArgs* args, int n, cudaStream_t stream) {
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  const RopeArgs& a = args[0];
  RopeKernelArgs k{};
  for (int i = 0; i < n; ++i) {
    k.t[i].in = static_cast<const uint4*>(args[i].in);
    k.t[i].out = static_cast<uint4*>(args[i].out);
    k.t[i].in_bs = args[i].in_batch_stride / 8;
    k.t[i].out_bs = args[i].out_batch_stride / 8;
  }
  k.n_tokens = (int)a.n_tokens;
  k.vec_per_tok = a.H * a.D / 8;
  k.vec_per_head = a.D / 8;
  k.gt = a.grid_t; k.gh = a.grid_h; k.gw = a.grid_w; k.t0 = a.t0;
  axis_split(a.D, &k.p_t, &k.p_h, &k.p_w);
  k.log2_base = (float)std::log2(a.base);
  const size_t smem = table_bytes(a);
  const bool fast = k.vec_per_tok % 32 == 0 && k.vec_per_tok / 32 <= kRopeFastMax && 32 % k.vec_per_head == 0;
  auto* kern = fast ? rope3d_fast_kernel : rope3d_kernel;
  static bool attr_done[64] = {false};
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (!attr_done[dev_id & 63]) {
    SAVGB_CUDA(cudaFuncSetAttribute(rope3d_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kRopeMaxTableBytes));
    SAVGB_CUDA(cudaFuncSetAttribute(rope3d_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kRopeMaxTableBytes));
    attr_done[dev_id & 63] = true;
  }
  // one wave: as many blocks as fit on the device at once, over all (batch, tensor) pairs
  int occ = 0;
  SAVGB_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kRopeThreads, smem));
  if (occ < 1) occ = 1;
  const int groups = (k.n_tokens + kRopeWarps - 1) / kRopeWarps;
  int per = occ * sms / (a.B * n);
  if (per < 1) per = 1;
  dim3 grid((unsigned)(groups < per ? groups : per), (unsigned)a.B, (unsigned)n);
  SAVGB_CUDA(launch_dependent(kern, grid, dim3(kRopeThreads), smem, stream, k));
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

int launch_rope(const RopeArgs& a, cudaStream_t stream) { return launch_rope_multi(&a, 1, stream); }

// Rotates two tensors of the same shape and grid (the chunk's q and k) in one launch.
int launch_rope_pair(const RopeArgs& a, const RopeArgs& b, cudaStream_t stream) {
  RopeArgs both[2] = {a, b};
  return launch_rope_multi(both, 2, stream);
}

}  // namespace savgb

extern "C" int rope3d_apply(const void* in, void* out, int B, int64_t n_tokens, int H, int D,
                            int grid_t, int grid_h, int grid_w, int t0, double base,
                            void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:rope3d_apply");
  clear_error();
  RopeArgs a{in, out, B, n_tokens, H, D, grid_t, grid_h, grid_w, t0, base,
             n_tokens * H * D, n_tokens * H * D};
  int rc = validate_rope(a);
  if (rc) return rc;
  return launch_rope(a, static_cast<cudaStream_t>(stream));
}
