// dt_topm_noalloc: the Top-M step for callers that cannot allocate device
// memory.  It runs the same kernel as dt_topm, but without a context: the
// kernel's scratch (per-chunk partial candidates and statistics, and the
// per-row arrival counters of the merge) lives in one fixed array of device
// memory that belongs to the library image, so a call performs no allocation.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace dt {

namespace {

// Upper bound of the scratch one call may use: rows * S * (8 M + 16) + 4 rows
// bytes, where S (the chunks per row) follows topm_plan.  Every GPU that loads
// the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_topm_scratch[kNoAllocScratchBytes];

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_topm_scratch
  int num_sms = 0;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: the device address of the
// scratch array (in host code the array's name is only a stand-in), the SM
// count, and the kernel's shared-memory attribute.
cudaError_t device_setup(DeviceSetup** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_topm_scratch);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = topm_prepare();
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<unsigned char*>(ptr);
    s.ready = true;
  }
  *out = &s;
  return cudaSuccess;
}

}  // namespace

}  // namespace dt

extern "C" dt_status dt_topm_noalloc(const float* logits, int rows, int V, int M, float T, int32_t* cand_tok,
                                     float* cand_base, float* rest_lse, void* stream) {
  using namespace dt;
  if (!logits || !cand_tok || !cand_base || !rest_lse) {
    set_last_error("dt_topm_noalloc: null pointer");
    return DT_ERR_INVALID_ARG;
  }
  if (rows < 1 || V < 1 || M < 1 || M > V || !(T > 0.0f)) {
    set_last_error("dt_topm_noalloc: need rows >= 1, 1 <= M <= V, T > 0");
    return DT_ERR_INVALID_ARG;
  }
  if (M > 512) {
    set_last_error("dt_topm_noalloc: M above 512");
    return DT_ERR_SHAPE;
  }
  DeviceSetup* dev = nullptr;
  cudaError_t e = device_setup(&dev);
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof(msg), "dt_topm_noalloc: device set-up failed: %s (%d)", cudaGetErrorString(e),
             static_cast<int>(e));
    set_last_error(msg);
    return DT_ERR_CUDA;
  }
  TopmParams p = {};
  p.logits = logits;
  p.V = V;
  p.rows = rows;
  p.M = M;
  p.T = T;
  topm_plan(p, dev->num_sms);
  if (const char* why = topm_unsupported(p)) {
    char msg[200];
    snprintf(msg, sizeof(msg), "dt_topm_noalloc: %d rows x %d logits with M=%d: %s", rows, V, M, why);
    set_last_error(msg);
    return DT_ERR_SHAPE;
  }
  // carve the scratch: partial ids / values, per-chunk statistics, row counters
  const size_t rs = static_cast<size_t>(rows) * p.S;
  size_t off = 0;
  const size_t o_id = off;
  off = align256(off + rs * M * 4);
  const size_t o_val = off;
  off = align256(off + rs * M * 4);
  const size_t o_max = off;
  off = align256(off + rs * 4);
  const size_t o_sum = off;
  off = align256(off + rs * 4);
  const size_t o_cnt = off;
  off = align256(off + rs * 4);
  const size_t o_kth = off;
  off = align256(off + rs * 4);
  const size_t o_done = off;
  off = align256(off + static_cast<size_t>(rows) * 4);
  if (off > kNoAllocScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "dt_topm_noalloc: %d rows x %d logits with M=%d need %zu scratch bytes, above the %zu-byte maximum",
             rows, V, M, off, kNoAllocScratchBytes);
    set_last_error(msg);
    return DT_ERR_SHAPE;
  }
  unsigned char* base = dev->scratch;
  p.part_id = reinterpret_cast<int*>(base + o_id);
  p.part_val = reinterpret_cast<float*>(base + o_val);
  p.part_max = reinterpret_cast<float*>(base + o_max);
  p.part_sum = reinterpret_cast<float*>(base + o_sum);
  p.part_cnt = reinterpret_cast<int*>(base + o_cnt);
  p.part_kth = reinterpret_cast<float*>(base + o_kth);
  p.row_done = reinterpret_cast<unsigned*>(base + o_done);
  p.cand_tok = cand_tok;
  p.cand_base = cand_base;
  p.rest_lse = rest_lse;
  p.status = nullptr;  // no context to hold a device status word
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the merge counts chunk arrivals per row from zero; the array keeps whatever
  // the previous call left, so clear the counters first
  e = cudaMemsetAsync(p.row_done, 0, static_cast<size_t>(rows) * 4, st);
  if (e == cudaSuccess) e = launch_topm(p, st);
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof(msg), "dt_topm_noalloc: launch failed: %s (%d)", cudaGetErrorString(e), static_cast<int>(e));
    set_last_error(msg);
    return DT_ERR_CUDA;
  }
  return DT_OK;
}
