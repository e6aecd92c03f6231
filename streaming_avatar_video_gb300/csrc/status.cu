// Status codes, thread-local messages, the device error word, device checks,
// tensor-map encoding and the host-side time grid.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <atomic>
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace savgb {

namespace {
thread_local char g_msg[512] = {0};

// One error word per device (a __device__ variable exists once per device
// that loads the module).
__device__ DeviceErrorWord g_dev_err;

constexpr int kMaxDevices = 64;
DeviceErrorWord* g_err_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};
std::mutex g_mu;
std::atomic<uint64_t> g_launches{0};
}  // namespace

void clear_error() { g_msg[0] = 0; }

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
std::mutex g_fault_mu;
int g_fault_kind = 0;
ArmedFault g_fault{-1, 0};
}  // namespace

bool take_fault(int kind, ArmedFault* out) {
  std::lock_guard<std::mutex> lk(g_fault_mu);
  if (g_fault_kind != kind) return false;
  *out = g_fault;
  g_fault_kind = 0;
  return true;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  const int code = (e == cudaErrorMemoryAllocation) ? SAVGB_ERR_OOM : SAVGB_ERR_CUDA;
  return fail(code, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int error_word(DeviceErrorWord** out) {
  int dev = 0;
  SAVGB_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(SAVGB_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    SAVGB_CUDA(cudaGetSymbolAddress(&p, g_dev_err));
    g_err_ptr[dev] = static_cast<DeviceErrorWord*>(p);
  }
  *out = g_err_ptr[dev];
  return SAVGB_OK;
}

int check_device(int* sm_count) {
  int dev = 0;
  SAVGB_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(SAVGB_ERR_UNSUPPORTED, "device index %d", dev);
  if (g_sm_count[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    SAVGB_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    SAVGB_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    SAVGB_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (major != 10 || minor != 3)
      return fail(SAVGB_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
    g_sm_count[dev] = sms;
  }
  if (sm_count) *sm_count = g_sm_count[dev];
  return SAVGB_OK;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  static cudaError_t once_err = cudaSuccess;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    once_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                cudaEnableDefault, &q);
    if (once_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn) return fail(SAVGB_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                       cudaGetErrorName(once_err));
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5];
  cuuint32_t e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), d, s, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SAVGB_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return SAVGB_OK;
}

// A kernel that waits on an mbarrier nothing arrives on, through the same
// bounded wait the library's kernels use, and reports the timeout in the
// device error word.  Used to test failure reporting without faulting.
__global__ void watchdog_selftest_kernel(DeviceErrorWord* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);
    abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!dev::mbar_wait(&bar, 0, &abort_flag, limit_ns)) {
      atomicOr(&err->flags, kErrSelfTestWait);
      atomicCAS(&err->where, 0u, 0xFFu);
    }
  }
  __syncthreads();
}

}  // namespace savgb

using namespace savgb;

extern "C" {

uint64_t savgb_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* savgb_status_string(int status) {
  switch (status) {
    case SAVGB_OK: return "SAVGB_OK";
    case SAVGB_ERR_INVALID_ARG: return "SAVGB_ERR_INVALID_ARG";
    case SAVGB_ERR_UNSUPPORTED: return "SAVGB_ERR_UNSUPPORTED";
    case SAVGB_ERR_ALIGNMENT: return "SAVGB_ERR_ALIGNMENT";
    case SAVGB_ERR_OOM: return "SAVGB_ERR_OOM";
    case SAVGB_ERR_CUDA: return "SAVGB_ERR_CUDA";
    case SAVGB_ERR_TIMEOUT: return "SAVGB_ERR_TIMEOUT";
    case SAVGB_ERR_STATE: return "SAVGB_ERR_STATE";
    default: return "SAVGB_ERR_UNKNOWN";
  }
}

const char* savgb_last_error(void) { return g_msg; }

int savgb_version(void) { return 100; }

int savgb_device_check(void* stream) {
  savgb::ApiRange api_range_("savgb:savgb_device_check");
  clear_error();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DeviceErrorWord* p = nullptr;
  int rc = error_word(&p);
  if (rc) return rc;
  DeviceErrorWord h{0, 0};
  SAVGB_CUDA(cudaMemcpy(&h, p, sizeof(h), cudaMemcpyDeviceToHost));
  if (h.flags == 0) return SAVGB_OK;
  const DeviceErrorWord zero{0, 0};
  SAVGB_CUDA(cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice));
  return fail(SAVGB_ERR_TIMEOUT, "a bounded device wait ran out (flags 0x%x:%s%s%s, wait code %u)",
              h.flags, (h.flags & kErrAttnWait) ? " chunk_attention" : "",
              (h.flags & kErrGemmWait) ? " out_proj_euler_step" : "",
              (h.flags & kErrSelfTestWait) ? " watchdog_selftest" : "", h.where);
}

int savgb_watchdog_selftest(uint64_t limit_ns, void* stream) {
  savgb::ApiRange api_range_("savgb:savgb_watchdog_selftest");
  clear_error();
  int rc = check_device(nullptr);
  if (rc) return rc;
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(SAVGB_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
  DeviceErrorWord* err = nullptr;
  if ((rc = error_word(&err))) return rc;
  watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

int savgb_arm_wait_fault(int kind, int index, uint64_t limit_ns) {
  clear_error();
  if (kind != SAVGB_FAULT_ATTENTION_K_TILE && kind != SAVGB_FAULT_WO_PAIR_RELAY)
    return fail(SAVGB_ERR_INVALID_ARG, "savgb_arm_wait_fault: unknown kind %d", kind);
  std::lock_guard<std::mutex> lk(g_fault_mu);
  if (index < 0) {
    if (g_fault_kind == kind) g_fault_kind = 0;
    return SAVGB_OK;
  }
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(SAVGB_ERR_INVALID_ARG, "savgb_arm_wait_fault: limit_ns must be in (0, 1e10]");
  g_fault_kind = kind;
  g_fault = ArmedFault{index, limit_ns};
  return SAVGB_OK;
}

int flow_time_grid(int steps, double shift, double* dt_out) {
  clear_error();
  if (steps < 1 || !(shift > 0.0) || !std::isfinite(shift) || dt_out == nullptr)
    return fail(SAVGB_ERR_INVALID_ARG, "flow_time_grid: steps >= 1, finite shift > 0, dt_out != NULL");
  auto warp = [&](int i) {
    const double sigma = 1.0 - static_cast<double>(i) / steps;
    return shift * sigma / (1.0 + (shift - 1.0) * sigma);
  };
  double prev = warp(0);
  for (int i = 0; i < steps; ++i) {
    const double next = warp(i + 1);
    dt_out[i] = prev - next;
    prev = next;
  }
  return SAVGB_OK;
}

}  // extern "C"
