// Host-side helpers shared by the library's translation units.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "savgb.h"

namespace savgb {

// Records a thread-local message for savgb_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Clears the thread-local message (called at the start of every entry point).
void clear_error();
// Counts one kernel the library enqueued (after the runtime accepted the launch);
// read through savgb_kernel_launches().
void note_launch();

// A named NVTX range around one C-ABI call, for profilers (ncu --nvtx
// filters kernels by it); with no tool attached it costs a few nanoseconds.
struct ApiRange {
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;
};
// Maps a CUDA runtime error to SAVGB_ERR_CUDA / SAVGB_ERR_OOM with a message.
int cuda_fail(cudaError_t e, const char* what);

#define SAVGB_CUDA(call)                                   \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return ::savgb::cuda_fail(e_, #call); \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device error word: bit flags set by kernels whose bounded waits ran out,
// plus the code of the wait that gave up first.  Lives in a file-scope
// __device__ variable (no allocation); this returns its device address on the
// current device.
struct DeviceErrorWord {
  unsigned int flags;
  unsigned int where;
};
enum : unsigned int {
  kErrAttnWait = 1u << 0,
  kErrGemmWait = 1u << 1,
  kErrSelfTestWait = 1u << 2,
};
int error_word(DeviceErrorWord** out);

// One-shot fault armed by savgb_arm_wait_fault (a failure-path test hook):
// the next launch of the kernel of `kind` takes it and disarms it.  The
// kernel then skips one arrival at `index` and bounds its waits by limit_ns.
struct ArmedFault {
  int index;
  uint64_t limit_ns;
};
bool take_fault(int kind, ArmedFault* out);

// Current device must be an sm_103 part (GB300); returns SAVGB_ERR_UNSUPPORTED
// otherwise.  Caches the SM count.
int check_device(int* sm_count);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// Internal launchers (all validate nothing: the entry points do that).
// Launches `kernel` as a programmatic dependent of the previous kernel of the
// stream (it may start while that one drains; the kernel itself waits with
// griddepcontrol.wait before touching memory that earlier work uses).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct RopeArgs {
  const void* in;
  void* out;
  int B;
  int64_t n_tokens;
  int H, D;
  int grid_t, grid_h, grid_w, t0;
  double base;
  int64_t in_batch_stride;   // elements between batches of `in`
  int64_t out_batch_stride;  // elements between batches of `out`
};
int validate_rope(const RopeArgs& a);
int launch_rope(const RopeArgs& a, cudaStream_t stream);
// Rotates two tensors of one shape and grid (a chunk's q and k) in one launch.
int launch_rope_pair(const RopeArgs& a, const RopeArgs& b, cudaStream_t stream);

struct AttnSeg {
  const void* k;
  const void* v;
  int64_t n;
};
int validate_attention(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                       int n_segs, const void* o);
// exact_softmax selects the instantiation with fp32 exponentials and exact row
// sums; so do a log-sum-exp output and a softmax scale above 1.25 x 1/sqrt(D).
int launch_attention(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                     int n_segs, float scale, void* o, float* lse, cudaStream_t stream,
                     bool exact_softmax = false);
// Grid of the (unrotated) queries for attention with RoPE of Q fused in.
struct QRope {
  int grid_t, grid_h, grid_w, t0;
  double base;
  // a cos/sin table from rope_q_table_build covering t in [tab_t_lo,
  // tab_t_lo + tab_t_n); null: launch_attention_qrope builds one per call
  const void* tab = nullptr;
  int tab_t_lo = 0, tab_t_n = 0;
};
int validate_qrope(const QRope& r, int64_t n_q, int D);
// The fused kernel's cos/sin table in global memory: [t rows | h | w] for
// n_t time values from t_lo and the whole h x w grid (bytes, a multiple of 16).
int64_t rope_q_table_bytes(int D, int n_t, int grid_h, int grid_w);
int rope_q_table_build(void* tab, int D, int t_lo, int n_t, int grid_h, int grid_w, double base,
                       cudaStream_t stream);
// Whether the fused kernel's shared-memory copy of the table fits.
bool qrope_fits(int D, int grid_t, int grid_h, int grid_w);
int launch_attention_qrope(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                           int n_segs, float scale, const QRope& rope, void* o, float* lse,
                           cudaStream_t stream, bool exact_softmax = false);

// QKV projection with the RoPE of q and k in the GEMM epilogue.
struct QkvArgs {
  const void* x_bf16;  // [B*n_tokens][H*D]
  const void* w_qkv;   // [3*H*D][H*D]
  void* q;
  void* k;
  void* v;
  void* k_tail;        // optional: unrotated k of the last n_tail tokens of each batch
  int64_t n_tail;
  int B;
  int64_t n_tokens;
  int H, D;
  int grid_t, grid_h, grid_w, t0;
  double base;
};
int validate_qkv(const QkvArgs& a);
int launch_qkv_rope(const QkvArgs& a, cudaStream_t stream);
int launch_to_bf16(const float* x, void* y, int64_t n, cudaStream_t stream);

int validate_out_proj(const void* o, const void* w, const float* bias, const float* x, int64_t M,
                      int hid_in, int hid_out, const float* v_out);
// x_copy (optional, fp32 like x, not with v_out): also receives the updated x.
int launch_out_proj_euler(const void* o, const void* w, const float* bias, float* x, int64_t M,
                          int hid_in, int hid_out, float dt, float* v_out, cudaStream_t stream,
                          float* x_copy = nullptr);

}  // namespace savgb
