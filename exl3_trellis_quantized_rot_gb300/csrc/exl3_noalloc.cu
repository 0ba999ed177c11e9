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
// threads) race on it, so order them on one stream.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tfx_exl3.h"
#include "exl3_kernels.cuh"

namespace tfx {
KernelSet kernels_b1();
KernelSet kernels_b2();
KernelSet kernels_b3();
KernelSet kernels_b4();
KernelSet kernels_b5();
KernelSet kernels_b6();
KernelSet kernels_b7();
KernelSet kernels_b8();
const void* rot_kernel_fn();
int report_error(int code, const char* msg);
}  // namespace tfx

namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
constexpr size_t kCounterBytes = 16u << 10;       // 4096 counters at the start of the array

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set up once).
int scratch_on_current_device(unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return tfx::report_error(TFX_EUNSUPPORTED, "device ordinal out of range");
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

tfx::KernelSet kernel_set(int bits) {
  switch (bits) {
    case 1: return tfx::kernels_b1();
    case 2: return tfx::kernels_b2();
    case 3: return tfx::kernels_b3();
    case 4: return tfx::kernels_b4();
    case 5: return tfx::kernels_b5();
    case 6: return tfx::kernels_b6();
    case 7: return tfx::kernels_b7();
    default: return tfx::kernels_b8();
  }
}

int launch_plain(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void* arg) {
  void* args[1] = {arg};
  cudaError_t e = cudaLaunchKernel(fn, grid, block, args, smem, s);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  return 0;
}

}  // namespace

extern "C" int tfx_exl3_linear_static(const tfx_exl3_weight* w, const void* x, int rows, void* y,
                                      cudaStream_t stream) {
  int S = 0, Wk = 0;
  int rc = tfx_exl3_plan(w, &S, &Wk);  // validates the descriptor
  if (rc) return rc;
  if (rows < 0 || !x || !y) return tfx::report_error(TFX_EINVAL, "rows < 0, or null x / y");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
    return tfx::report_error(TFX_EALIGN, "x and y must be 16-byte aligned");
  if (rows == 0) return 0;

  const int K = w->K, N = w->N, NB = N / 128;
  const int passes = (rows + tfx::kRowsPerPass - 1) / tfx::kRowsPerPass;
  const int rp = rows < tfx::kRowsPerPass ? rows : tfx::kRowsPerPass;
  const size_t counter_bytes = (size_t)passes * NB * sizeof(int);
  const size_t xr_bytes = (size_t)rows * K * 2;
  const size_t partial_bytes = (size_t)passes * S * rp * N * sizeof(float);
  const size_t need = kCounterBytes + align256(xr_bytes) + partial_bytes;
  if (counter_bytes > kCounterBytes || need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "tfx_exl3_linear_static needs %zu bytes of scratch (%zu of counters) for %d rows of %dx%d; "
             "the static scratch holds %zu bytes (%zu of counters)",
             need, counter_bytes, rows, K, N, kStaticScratchBytes, kCounterBytes);
    return tfx::report_error(TFX_EUNSUPPORTED, msg);
  }
  unsigned char* base = nullptr;
  rc = scratch_on_current_device(&base);
  if (rc) return rc;
  int* counters = reinterpret_cast<int*>(base);
  __half* xr = reinterpret_cast<__half*>(base + kCounterBytes);
  float* partial = reinterpret_cast<float*>(base + kCounterBytes + align256(xr_bytes));

  // the array keeps whatever the last call left: start this call's counters at zero
  cudaError_t e = cudaMemsetAsync(counters, 0, counter_bytes, stream);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));

  tfx::RotArgs ra = {};
  ra.x = x;
  ra.count = 1;
  ra.rows = rows;
  ra.K = K;
  ra.act = w->act;
  ra.suh[0] = reinterpret_cast<const __half*>(w->suh);
  ra.xr[0] = xr;
  const long long items = (long long)rows * (K / 128);
  rc = launch_plain(tfx::rot_kernel_fn(), dim3((unsigned)((items + 7) / 8)), dim3(256), 0, stream, &ra);
  if (rc) return rc;

  // kernel family: 1..16 rows decode-rows (8 warps), otherwise mid-rows (16 warps)
  const tfx::KernelSet ks = kernel_set(w->bits);
  const void* fn;
  int wpc, nr;
  if (rows <= 16) {
    fn = rp <= 8 ? ks.linear_rows[0] : ks.linear_rows[1];
    wpc = 8;
    nr = rp <= 8 ? 1 : 2;
  } else if (rp <= 32) {
    fn = ks.linear_mid[1], wpc = 16, nr = 4;
  } else if (rp <= 64) {
    fn = ks.linear_mid[2], wpc = 16, nr = 8;
  } else {
    fn = ks.linear_mid[3], wpc = 16, nr = 16;
  }
  tfx::LinearArgs la = {};
  la.count = 1;
  la.K = K;
  la.TK = K / 16;
  la.rows = rows;
  la.passes = passes;
  la.rp = rp;
  la.act = w->act;
  tfx::Member& m = la.m[0];
  m.trellis = w->trellis;
  m.stride = w->tile_row_stride;
  m.svh = reinterpret_cast<const __half*>(w->svh);
  m.xr = xr;
  m.y = y;
  m.partial = partial;
  m.counters = counters;
  m.N = N;
  m.NB = NB;
  m.S = S;
  m.Wk = Wk;
  m.TC = wpc / Wk > 8 ? 8 : wpc / Wk;
  m.subs = 8 / m.TC;
  m.cta_begin = 0;
  const long long ctas = (long long)NB * m.subs * S * passes;
  const size_t smem = (size_t)wpc * nr * 8 * 16 * sizeof(float);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  }
  return launch_plain(fn, dim3((unsigned)ctas), dim3(wpc * 32), smem, stream, &la);
}
