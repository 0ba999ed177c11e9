// tfx_exl3_linear_static: the linear layer with its scratch in a fixed,
// file-scope device array instead of memory obtained by tfx_exl3_reserve.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at
// the point where they run the layer — for example code that runs inside a
// host callback or a driver-managed context where allocation is forbidden,
// plugins whose host application owns all device memory, or runtimes that
// must not allocate after start-up. They pass x and y, and the library uses
// a static scratch area every GPU loading the library keeps until exit.
//
// The scratch array is a host-side stand-in in host code: its device address
// comes from cudaGetSymbolAddress, taken once per device (with that device
// current) on the first call made on that device. Make that first call before
// any stream capture. All calls share the one array and see what the last
// call left there; calls that overlap on the GPU (other streams, other
// threads) race on it, so order them on one stream. The stream must belong
// to the current device.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tfx_exl3.h"
#include "exl3_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
constexpr size_t kCounterBytes = 16u << 10;       // 4096 counters at the start of the array

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set up once),
// after checking that `stream` belongs to that device.
int scratch_on_current_device(cudaStream_t stream, unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return tfx::report_error(TFX_EUNSUPPORTED, "device ordinal out of range");
  if (stream) {
    int sdev = -1;
    e = cudaStreamGetDevice(stream, &sdev);
    if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
    if (sdev != dev)
      return tfx::report_error(TFX_EINVAL, "the stream belongs to another device than the current one");
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) return tfx::report_error(TFX_ECUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_dev_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_dev_ptr[dev]);
  return 0;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

extern "C" int tfx_exl3_linear_static(const tfx_exl3_weight* w, const void* x, int rows, void* y,
                                      cudaStream_t stream) {
  int C = 0, tiles = 0;
  int rc = tfx_exl3_plan(w, &C, &tiles);  // validates the descriptor
  if (rc) return rc;
  if (rows < 0 || !x || !y) return tfx::report_error(TFX_EINVAL, "rows < 0, or null x / y");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
    return tfx::report_error(TFX_EALIGN, "x and y must be 16-byte aligned");
  if (rows == 0) return 0;

  const size_t counter_bytes = tfx::counter_bytes_needed(w, rows);
  const size_t xf_bytes = tfx::xf_bytes_needed(w, rows);
  const size_t partial_bytes = tfx::partial_bytes_needed(w, rows);
  const size_t need = kCounterBytes + align256(xf_bytes) + partial_bytes;
  if (counter_bytes > kCounterBytes || need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "tfx_exl3_linear_static needs %zu bytes of scratch (%zu of counters) for %d rows of %dx%d; "
             "the static scratch holds %zu bytes (%zu of counters)",
             need, counter_bytes, rows, w->K, w->N, kStaticScratchBytes, kCounterBytes);
    return tfx::report_error(TFX_EUNSUPPORTED, msg);
  }
  unsigned char* base = nullptr;
  rc = scratch_on_current_device(stream, &base);
  if (rc) return rc;
  tfx::Scratch sc = {};
  sc.err = reinterpret_cast<int*>(base);
  sc.counters[0] = reinterpret_cast<int*>(base) + tfx::kErrorInts;
  sc.xf[0] = reinterpret_cast<uint2*>(base + kCounterBytes);
  sc.partial[0] = reinterpret_cast<float*>(base + kCounterBytes + align256(xf_bytes));

  // the array keeps whatever the last call left: clear the device error word
  // and exactly this call's counters (counter_bytes covers both, from the
  // start of the array)
  cudaError_t e = cudaMemsetAsync(base, 0, counter_bytes, stream);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));

  tfx_exl3_weight wc = *w;
  tfx_exl3_weight* ws[1] = {&wc};
  void* ys[1] = {y};
  return tfx::launch_layer(ws, 1, x, rows, ys, nullptr, nullptr, stream, sc, 0);
}
