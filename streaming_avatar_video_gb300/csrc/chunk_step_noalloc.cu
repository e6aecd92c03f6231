// chunk_step_noalloc: one chunk denoising step that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a plugin hosted by a serving runtime
// that owns every device allocation through its own pool and gives plugins no
// allocator, or a latency-critical loop in which an allocation (with the
// device synchronisation cudaMalloc/cudaFree may imply) is not allowed once
// the session runs.  Those callers cannot create a chunk_stream handle, whose
// arena is allocated at create.  This entry point runs the same step as
// chunk_stream_step (RoPE of k, attention over the caller's context segments
// plus the chunk with the RoPE of q inside the kernel, W_o with the Euler
// update; or, when the kernel's cos/sin table does not fit, RoPE of q and k
// in one launch and the plain attention) and keeps its intermediates -
// rotated k, the attention output and the table, or rotated q in its place -
// in one file-scope __device__ array of a fixed size instead.  The table is
// rebuilt by every call.
//
// The array exists once per device that loads this library and is held until
// the process exits.  Its device address is looked up once per device (with
// that device current) on the first call made on that device; make that first
// call before any stream capture.  Every call shares the array: calls that
// overlap on the GPU (different streams, or different host threads on one
// device) race on it.  Each call writes every scratch element it later reads,
// so nothing needs clearing between calls.
#include <cmath>
#include <mutex>

#include "common.h"

namespace savgb {
namespace {

constexpr size_t kScratchBytes = SAVGB_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_step_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  SAVGB_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDev) return fail(SAVGB_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "chunk_step_noalloc: cudaGetSymbolAddress(scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SAVGB_OK;
}

}  // namespace
}  // namespace savgb

extern "C" int chunk_step_noalloc(const void* q, const void* k, const void* v,
                                  const savgb_kv_segment* context, int n_context, const void* w_o,
                                  const float* bias, float* x, float dt, int B, int H, int D, int F,
                                  int grid_h, int grid_w, double rope_base, float softmax_scale,
                                  void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:chunk_step_noalloc");
  clear_error();
  if (!q || !k || !v || !w_o || !x) return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: null argument");
  if (n_context < 0 || n_context > 2 || (n_context > 0 && !context))
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: 0 to 2 context segments");
  if (B < 1 || B > 65535 || H < 1 || H > 65535 || F < 1 || grid_h < 1 || grid_w < 1)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: B, H in [1, 65535]; F, grid_h, grid_w >= 1");
  if (F > 4096 || grid_h > 4096 || grid_w > 4096)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: F, grid_h and grid_w must be <= 4096");
  if (D != 64 && D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_step_noalloc: head_dim %d (64 or 128)", D);
  if (!std::isfinite(dt)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: dt must be finite");
  // every size below is bounded now: n <= 2^36, hid <= 2^24, B < 2^16
  const int64_t n = (int64_t)F * grid_h * grid_w;
  const int64_t hid = (int64_t)H * D;
  if (hid > (1 << 24) || hid % 16)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_step_noalloc: H*D = %lld must be a multiple of 16 and at most 2^24",
                (long long)hid);
  // the fused form keeps the q RoPE table where the unfused one keeps rotated q;
  // the sizes are summed in double, which is exact here and cannot overflow
  const bool fused = qrope_fits(D, F, grid_h, grid_w);
  const double tensor_d = std::ceil((double)B * (double)n * (double)hid * 2.0 / 256.0) * 256.0;
  const double third_d = fused ? std::ceil((double)rope_q_table_bytes(D, F, grid_h, grid_w) / 256.0) * 256.0 : tensor_d;
  const double need = 2.0 * tensor_d + third_d;
  if (need > (double)kScratchBytes)
    return fail(SAVGB_ERR_INVALID_ARG,
                "chunk_step_noalloc: the step needs %.0f bytes of scratch (rotated k, attention output and the "
                "q RoPE table or rotated q), more than the fixed %zu bytes; use a chunk_stream handle for "
                "larger chunks",
                need, kScratchBytes);
  const int64_t tensor_bytes = (int64_t)tensor_d;
  // shapes and pointers of the three launches, checked before any launch
  RopeArgs aq{q, (void*)16, B, n, H, D, F, grid_h, grid_w, 0, rope_base, n * hid, n * hid};
  RopeArgs ak = aq;
  ak.in = k;
  int rc = validate_rope(aq);
  if (!rc) rc = validate_rope(ak);
  if (rc) return rc;
  AttnSeg segs[3] = {};
  for (int i = 0; i < n_context; ++i)
    segs[i] = AttnSeg{context[i].k, context[i].v, context[i].n_tokens};
  segs[n_context] = AttnSeg{(const void*)16, v, n};
  if ((rc = validate_attention((const void*)16, B, n, H, D, segs, n_context + 1, (const void*)16))) return rc;
  if ((rc = validate_out_proj((const void*)16, w_o, bias, x, (int64_t)B * n, (int)hid, (int)hid, nullptr)))
    return rc;
  if ((rc = check_device(nullptr))) return rc;

  void* base = nullptr;
  if ((rc = scratch_address(&base))) return rc;
  unsigned char* p = static_cast<unsigned char*>(base);
  void* k_rot = p;
  void* o = p + tensor_bytes;
  void* third_buf = p + 2 * tensor_bytes;  // the table (fused) or rotated q
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  ak.out = k_rot;
  segs[n_context].k = k_rot;
  if (fused) {
    if ((rc = rope_q_table_build(third_buf, D, 0, F, grid_h, grid_w, rope_base, st))) return rc;
    if ((rc = launch_rope(ak, st))) return rc;
    QRope r{F, grid_h, grid_w, 0, rope_base};
    r.tab = third_buf;
    r.tab_t_lo = 0;
    r.tab_t_n = F;
    if ((rc = launch_attention_qrope(q, B, n, H, D, segs, n_context + 1, softmax_scale, r, o, nullptr, st)))
      return rc;
  } else {
    aq.out = third_buf;
    if ((rc = launch_rope_pair(aq, ak, st))) return rc;
    if ((rc = launch_attention(third_buf, B, n, H, D, segs, n_context + 1, softmax_scale, o, nullptr, st)))
      return rc;
  }
  return launch_out_proj_euler(o, w_o, bias, x, (int64_t)B * n, (int)hid, (int)hid, dt, nullptr, st);
}
