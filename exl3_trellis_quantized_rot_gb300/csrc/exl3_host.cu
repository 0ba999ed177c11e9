// Host side of the tfx_exl3 C ABI: validation, plan, scratch reservation,
// kernel choice and launches. No CPU fallback exists: every step of the
// layer runs in the kernels of exl3_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/tfx_exl3.h"
#include "exl3_internal.h"
#include "exl3_tc.cuh"

namespace tfx {
KernelSet kernels_b1();
KernelSet kernels_b2();
KernelSet kernels_b3();
KernelSet kernels_b4();
KernelSet kernels_b5();
KernelSet kernels_b6();
KernelSet kernels_b7();
KernelSet kernels_b8();
}  // namespace tfx

namespace tfx {
// Rotation of x for up to 3 sign vectors: xf_m = fp16(Hn(suh_m o x)) per
// 128-block, written in B-fragment order (xf_index) for the decode-rows kernel
// or in core-matrix order (xc_byte) for the tensor-core kernel. One warp per
// (row, 128-block); x is read once; rows rows..rows_pad-1 are written as zero.
__global__ void __launch_bounds__(256) rot_kernel(const __grid_constant__ RotArgs a) {
  // wait first; the linear kernel may launch once every warp has stored its
  // block (a warp with no block has exited, which counts the same): an early
  // trigger lets the linear kernel's CTAs hold SM resources while the
  // rotation still runs (measured slower inside graphs)
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nblk = a.K / 128;
  if (item >= (long long)a.rows_pad * nblk) return;
  const int r = (int)(item / nblk);
  const int b = (int)(item % nblk);
  // every member's suh is requested together with x: inside the member loop
  // each load would wait for the previous member's stores (the compiler cannot
  // move a load across stores that may alias it)
  uint2 su[3];
#pragma unroll
  for (int m = 0; m < 3; m++)
    if (m < a.count) su[m] = rot_suh(a, m, b, lane);
  float xv[4];
  rot_load(a, r, b, lane, xv);
#pragma unroll
  for (int m = 0; m < 3; m++) {
    if (m >= a.count) break;
    __half2 h[2];
    rot_member_su(su[m], lane, xv, h);
    if (a.layout == 0) {
      rot_store_frag(a, m, r, b, lane, h);
    } else {
      // the lane's 4 values are k%8 = 4*(lane%2) .. +3 of one core-matrix row: one 8-byte store
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&h[0]);
      o.y = *reinterpret_cast<uint32_t*>(&h[1]);
      *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(a.xf[m]) + xc_byte(r, 128 * b + 4 * lane, a.K, a.rp_tc, a.rows_pad)) = o;
    }
  }
  griddep_launch();
}

__global__ void __launch_bounds__(256) tc_combine_kernel(const __grid_constant__ CombineArgs ca) {
  griddep_wait();
  griddep_launch();
  const LinearArgs& a = ca.la;
  long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  int mi = 0;
  while (mi < a.count && w >= ca.items[mi]) {
    w -= ca.items[mi];
    mi++;
  }
  if (mi >= a.count) return;
  combine_item(a, a.m[mi], (int)(w / a.m[mi].NB), (int)(w % a.m[mi].NB), ca.RP, lane);
}

}  // namespace tfx

namespace {
using tfx::kRowsPerPass;

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(TFX_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- driver hooks

int rt_alloc(void** p, size_t bytes, cudaStream_t s) { return cudaMallocAsync(p, bytes, s) == cudaSuccess ? 0 : -1; }
int rt_free(void* p, cudaStream_t s) { return cudaFreeAsync(p, s) == cudaSuccess ? 0 : -1; }
int rt_memset0(void* p, size_t bytes, cudaStream_t s) { return cudaMemsetAsync(p, 0, bytes, s) == cudaSuccess ? 0 : -1; }

// Allocation hooks of reserve/release (the CUDA runtime, or a test's fake);
// swapped and read under a lock so that a test hook never tears a call.
std::mutex g_drv_mu;
tfx_exl3_driver g_drv_hooks = {rt_alloc, rt_free, rt_memset0};
tfx_exl3_driver drv() {
  std::lock_guard<std::mutex> lk(g_drv_mu);
  return g_drv_hooks;
}

int env_variant() {
  const char* v = getenv("TFX_EXL3_VARIANT");
  if (!v) return 0;
  if (!strcmp(v, "rows")) return 1;
  if (!strcmp(v, "mid")) return 2;
  if (!strcmp(v, "warp")) return 3;
  if (!strcmp(v, "warp_global")) return 4;
  return 0;
}
// Programmatic dependent launch: 0 off, 1 on every kernel, 2 (the default)
// automatic: on the rotation launch and on the decode-rows linear launch that
// follows it, and on the combine launch after a decode-rows launch that folds
// through slabs (measured on GB300: the q/k/v group at 16 rows 22.6 -> 21.8
// us), nowhere else. Measured on GB300 inside CUDA graphs (calls back
// to back, K = 5120, 4-bit): with it on every kernel a 1-row 5120 x 5120 call
// (one fused kernel, no rotation launch) takes 14.3 us against 13.0 without;
// on the rotation and decode-rows launches of 7- and 16-row calls it saves
// 3-5 % (16 rows: 16.7 -> 16.2 us, q/k/v group 24.3 -> 23.6 us).
// TFX_EXL3_PDL=0 or 1 overrides the default.
int env_pdl() {
  const char* v = getenv("TFX_EXL3_PDL");
  if (v && !strcmp(v, "0")) return 0;
  if (v && !strcmp(v, "1")) return 1;
  return 2;
}
// Process-wide switches: read by every call, written by the set_* hooks.
std::atomic<int> g_variant{env_variant()};
thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
std::atomic<int> g_pdl{env_pdl()};
std::atomic<long long> g_spin{tfx::kSpinClocks};
std::atomic<long long> g_launches{0};  // kernels enqueued (or captured) through the library

// ---------------------------------------------------------------- per-weight state

struct Priv {
  uint2* xf = nullptr;
  size_t xf_bytes = 0;
  float* partial = nullptr;
  size_t partial_bytes = 0;
  int* counters = nullptr;
  size_t counter_bytes = 0;
  float* lev = nullptr;  // tensor-core kernel: per-CTA slots for the deepest chunk-tree levels
  size_t lev_bytes = 0;
  int max_rows = 0;
  int64_t allocs = 0, memsets = 0;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const tfx_exl3_weight* w) {
  if (!w) return fail(TFX_EINVAL, "null weight");
  if (w->K <= 0 || w->N <= 0 || w->K % 128 || w->N % 128)
    return fail(TFX_EINVAL, "K=%d and N=%d must be positive multiples of 128", w->K, w->N);
  if (w->bits < 1 || w->bits > 8) return fail(TFX_EINVAL, "bits=%d outside 1..8", w->bits);
  if (w->act != TFX_F16 && w->act != TFX_BF16) return fail(TFX_EINVAL, "act=%d", w->act);
  if (!w->trellis || !w->suh || !w->svh) return fail(TFX_EINVAL, "null trellis/suh/svh");
  if (w->tile_row_stride < (int64_t)(w->N / 16) * 8 * w->bits)
    return fail(TFX_EINVAL, "tile_row_stride %lld below the weight's own %lld words",
                (long long)w->tile_row_stride, (long long)(w->N / 16) * 8 * w->bits);
  if (w->tile_row_stride % 4)
    return fail(TFX_EALIGN, "tile_row_stride %lld is not a multiple of 4 words (16 bytes)",
                (long long)w->tile_row_stride);
  if (!aligned16(w->trellis) || !aligned16(w->suh) || !aligned16(w->svh))
    return fail(TFX_EALIGN, "trellis/suh/svh must be 16-byte aligned");
  return 0;
}


// SMs of the current device (152 on GB300; also the answer when no device is visible).
int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Decode rows: warp groups per column (GW) and chunks per warp (G). GW*G
// chunks form one CTA's subtree; G grows while the launch keeps at least
// 4 CTAs per SM (launch shape only; the bits do not depend on it).
int rows_gw(int C) { return C < tfx::kRowsGW ? C : tfx::kRowsGW; }
int rows_group(int TN, int C, int rows) {
  if (rows > 16) return 1;  // 32- and 64-row tiles park no tree levels
  const int gw = rows_gw(C);
  const long long want = 4LL * sm_count();
  int g = 1;
  while (2 * g <= (1 << tfx::kRowsMaxLog2G) && gw * 2 * g <= C &&
         (long long)(TN / tfx::kRowsTC) * (C / (gw * 2 * g)) >= want)
    g *= 2;
  return g;
}

struct KernelTable {
  tfx::KernelSet ks[9];
  KernelTable() {
    ks[1] = tfx::kernels_b1();
    ks[2] = tfx::kernels_b2();
    ks[3] = tfx::kernels_b3();
    ks[4] = tfx::kernels_b4();
    ks[5] = tfx::kernels_b5();
    ks[6] = tfx::kernels_b6();
    ks[7] = tfx::kernels_b7();
    ks[8] = tfx::kernels_b8();
  }
};
// Built once, on first use (a function-local static: thread-safe initialisation).
const tfx::KernelSet& kernels(int bits) {
  static const KernelTable table;
  return table.ks[bits];
}

// Launch with an optional programmatic dependency on the previous kernel of
// the stream and an optional 1-D cluster of `cluster` CTAs.
int launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void* arg, bool pdl, int cluster = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    na++;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  void* args[1] = {arg};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return 0;
}

// The linear kernel family for `rows` rows.
enum Kind { kRowsCta = 0, kRowsWarp = 1, kTensor = 2 };
struct Family {
  const void* fn;
  int wpc;   // warps per CTA
  int ncol;  // tile-columns per warp (warp-granular kernel)
  Kind kind;
  int nr;    // 8-row groups of the decode-rows row tile
  // decode-rows families: x in m16n8k16 fragment order, one pass
  bool rows() const { return kind == kRowsCta || kind == kRowsWarp; }
};

int row_tile(int rows) { return rows <= 8 ? 0 : rows <= 16 ? 1 : rows <= 32 ? 2 : 3; }

// Calls of at most this many rows skip the rotation kernel: the decode-rows
// kernel rotates each CTA's chunk of x itself.
constexpr int kFuseRotRows = 4;
constexpr long long kFuseRotWeights = 64LL << 20;
// Decode-rows launches of more clusters than this arrive early on the closing
// cluster barrier (LinearArgs::early_arrive).
constexpr long long kEarlyArriveClusters = 128;
// auto sends calls of up to this many rows to the decode-rows kernel.
constexpr int kAutoRowsMax = 16;
// How the decode-rows kernel folds a block's chunk sums (LinearArgs::fold_mode).
// In the block's cluster every CTA waits at the cluster barrier for its
// slowest chunk while holding its SM slot; with many blocks that wait is what
// the next clusters queue behind. Global slabs folded by the combine kernel
// (one warp per row and block) free every CTA as soon as its chain is done.
// Measured on GB300 (graph-replayed, K = 5120; cluster / counter / combine):
//   40 blocks, 1 / 4 / 8 / 16 rows: 12.6 / 13.9 / 14.2 / 16.1 us with the
//     cluster, 14.1 / 16.7 / 20.8 / 29.8 with the counter, 13.9 / 15.8 / 15.6
//     / 17.1 with the combine kernel;
//   the q/k/v group (64 blocks) at 1 / 7 / 16 rows: 17.3 / 20.0 / 23.3 with
//     the cluster, 18.2 / 19.8 / 21.9 with the combine kernel;
//   272 blocks at 1 / 4 / 8 rows: 53.8 / 54.6 / 55.2, 49.6 / 51.4 / 55.0,
//     49.0 / 49.3 / 50.0; gate+up at 16 rows 65.8 against 58.5 combined;
//   768 blocks (6-bit), 1 / 4 / 8 rows: 177 / 178 / 180, 149 / 152 / 158,
//     147 / 148 / 151; the 6-bit LM head (1940 blocks): 433 / 435 / 438,
//     358 / 364 / 374, 352 / 361 / 371.
// The last-arriver counter form (PR #1475) is the forced variant 4 (up to
// kFoldCounterRows rows).
constexpr int kFoldCounterRows = 8;
int fold_mode_for(int rows, long long blocks) {
  if (g_variant.load(std::memory_order_relaxed) == 4 && rows <= kFoldCounterRows) return tfx::kFoldCounter;
  if (blocks > 128 || (blocks > 48 && rows > 8)) return tfx::kFoldCombine;
  return tfx::kFoldCluster;
}

// Kernel choice. auto: up to 16 rows the warp-granular decode-rows kernel,
// above that the persistent tensor-core kernel (measured on GB300, 4-bit,
// K = 5120, graph-replayed calls, decode-rows against tensor core: 5120 x 5120
// at 12 / 16 / 20 / 32 rows 15.4 / 16.1 / 25.2 / 25.8 us against 25.1 / 25.1 /
// 25.6 / 25.9; the q/k/v group 21.8 / 22.3 / 32.9 / 34.5 against 30.2 / 30.4 /
// 31.0 / 31.3; gate+up 58.4 / 58.6 / 111.6 / 118.3 against 88.8 / 89.5 / 90.2 /
// 91.2: above 16 rows the decode-rows kernel's row tile doubles its MMAs per
// decoded tile). The other variants force a family where it serves the row
// count (all give the same bytes).
Family pick(int bits, int rows) {
  const tfx::KernelSet& ks = kernels(bits);
  const int i = rows <= tfx::kRowsMaxRows ? row_tile(rows) : 0;
  const int ncol = i < 2 ? 2 : 1;  // must match the instantiations in exl3_bits.cu
  const Family warpk{ks.linear_warp[i], tfx::warp_cta_warps(ncol), ncol, kRowsWarp, 1 << i};
  const Family rowsk{ks.linear_rows[i], tfx::kRowsTC * tfx::kRowsGW, 1, kRowsCta, 1 << i};
  const Family tc{ks.linear_tc, tfx::kTcThreads / 32, 0, kTensor, 0};
  switch (g_variant.load(std::memory_order_relaxed)) {
    case 1: return rows <= tfx::kRowsMaxRows ? rowsk : tc;
    case 2: return tc;
    case 3:
    case 4: return rows <= tfx::kRowsMaxRows ? warpk : tc;
    default:
      if (rows <= kAutoRowsMax) return warpk;
      return tc;
  }
}

// Tensor-core kernel: rows per pass, and chunks per work unit (G). A pass is
// up to 128 rows (the MMA's N). With level scratch (a reserved weight) every
// unit of a call above 128 rows holds all C chunks of a 128-row pass: TMEM
// keeps the two pairs of accumulator regions and the first chunk-tree levels,
// deeper levels go to the scratch, so each weight is decoded once per 128
// rows. Without it (the static-scratch entry point) passes above 128 rows are
// 64 rows, where all levels fit in TMEM. Up to 128 rows, G (at least 2: a unit
// holds whole chunk pairs) is the power of two that minimises the persistent
// CTAs' critical path, ceil(units / SMs) unit lengths plus a fixed per-unit
// cost of 16 k-steps (pipeline fill and fold; measured on GB300 by forcing
// each G), among those whose levels fit TMEM when no level scratch is given. Launch shape only: the bits do not depend
// on the pass size or on G.
int tc_rows_per_pass(int rows, bool spill) {
  return rows <= tfx::kTcRowsMax || spill ? tfx::kTcRowsMax : tfx::kTcRowsNoSpill;
}
int tc_passes(int rows, bool spill) {
  const int rp = tc_rows_per_pass(rows, spill);
  return (rows + rp - 1) / rp;
}
// Chunk-tree levels above the pairs that TMEM holds next to the two pairs of
// accumulator regions of nm columns (at most 3, the levels of 8 pairs).
int tc_tmem_levels(int nm) {
  const int l = 512 / nm - 4;
  return l < tfx::kTcMaxLevels ? l : tfx::kTcMaxLevels;
}
int tc_group(long long blocks, int rows, int C, int TK, long long S, bool spill) {
  if (rows > tfx::kTcRowsMax) return C;
  const int nm = (rows + 15) / 16 * 16;
  int best = 2;
  long long best_cost = -1;
  for (int g = C; g >= 2; g /= 2) {
    // a unit holds whole chunk pairs: log2(g) - 1 levels above them
    const int lg = __builtin_ctz(g);
    if (lg - 1 > tc_tmem_levels(nm) + (spill ? tfx::kTcSpillLevels : 0)) continue;
    const long long units = blocks * (C / g);
    const long long cost = (units + S - 1) / S * ((long long)TK * g / C + 16);
    if (best_cost < 0 || cost < best_cost) {
      best = g;
      best_cost = cost;
    }
  }
  return best;
}

// Opt in to more than the default 48 KB of shared memory once per kernel and size.
int set_smem(const void* fn, size_t smem) {
  static thread_local const void* last_fn[16] = {};
  static thread_local size_t last_sz[16] = {};
  if (smem < 32 * 1024) return 0;
  for (int i = 0; i < 16; i++)
    if (last_fn[i] == fn && last_sz[i] >= smem) return 0;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  static thread_local int next = 0;
  last_fn[next] = fn;
  last_sz[next] = smem;
  next = (next + 1) % 16;
  return 0;
}

// Shared-memory carveout (percent of the maximum) for a kernel; the call is
// skipped when the kernel already has that value.
int set_carveout(const void* fn, int pct) {
  static thread_local const void* fns[32] = {};
  static thread_local int vals[32] = {};
  int slot = -1;
  for (int i = 0; i < 32; i++) {
    if (fns[i] == fn) {
      if (vals[i] == pct) return 0;
      slot = i;
      break;
    }
    if (!fns[i] && slot < 0) slot = i;
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, pct);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(carveout)");
  if (slot >= 0) {
    fns[slot] = fn;
    vals[slot] = pct;
  }
  return 0;
}

// Allow clusters above the portable 8 CTAs for a kernel, once per kernel.
int allow_big_clusters(const void* fn) {
  static thread_local const void* done[64] = {};
  for (int i = 0; i < 64; i++) {
    if (done[i] == fn) return 0;
    if (!done[i]) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster size)");
      done[i] = fn;
      return 0;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e == cudaSuccess ? 0 : cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster size)");
}

// cuTensorMapEncodeTiled from the driver the runtime loaded (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// The trellis of w as a 2-D tensor of uint32 words: x = word within a tile row
// (the view's N/16 * 8 * bits words), y = tile row (K/16), row pitch = the
// tile-row stride; boxes of `box_words` x `box_rows`.
int encode_trellis_map(const tfx_exl3_weight* w, int box_words, int box_rows, CUtensorMap* tm) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(TFX_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)(w->N / 16) * 8 * w->bits, (cuuint64_t)(w->K / 16)};
  cuuint64_t strides[1] = {(cuuint64_t)w->tile_row_stride * 4};
  cuuint32_t box[2] = {(cuuint32_t)box_words, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(w->trellis), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TFX_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return 0;
}

// Warp-granular kernel: how the chunk's operands are staged in shared memory,
// within 40 KB per CTA. The x fragments of the whole chunk form one stage
// loaded once when they take at most half of it; the trellis words are one
// box per warp when they fit the rest, else two boxes of H rows in flight
// (refilled as they are used). When even x does not fit, x and words share
// H-row boxes, two in flight. Measured on GB300: staging the whole 5120-wide
// chunk at once (30 KB per CTA at 16 rows) beats smaller boxes that would let
// all 64 clusters of a q/k/v group be resident at once (25 KB: 68 resident
// clusters against 54 at 30 KB), because the refills cost more than the
// second partial wave.
struct WarpStaging {
  int H, R, XH, x_whole;
};
WarpStaging warp_staging(int K, int bits, int ncol, int nr, long long clusters) {
  const int C = tfx::chunks_of(K), TK = K / 16;
  const int nmax = (TK + C - 1) / C;
  (void)clusters;
  const int budget = 40 * 1024 - 128;
  const int wrow = tfx::warp_cta_warps(ncol) * tfx::warp_row_bytes(bits, ncol);  // words of one tile row, all warps
  const int xrow = nr * 256;                                                       // x of one tile row
  WarpStaging st{};
  auto split = [&](int rows_cap) {
    int h = rows_cap < 1 ? 1 : rows_cap;
    if (h > nmax) h = nmax;
    const int nb = (nmax + h - 1) / h;
    return (nmax + nb - 1) / nb;
  };
  if (nmax * xrow <= budget / 2) {
    st.x_whole = 1;
    st.XH = nmax;
    const int left = budget - nmax * xrow;
    if (nmax * wrow <= left) {
      st.H = nmax;
      st.R = 1;
    } else {
      st.H = split(left / (2 * wrow));
      st.R = 2;
    }
  } else {
    st.x_whole = 0;
    st.H = split(budget / (2 * (wrow + xrow)));
    st.R = 2;
    st.XH = st.H;
  }
  return st;
}

// Record a measurement event on `s`; inside a stream capture it becomes an
// event-record node of the graph (external record), so that the event can be
// timed when the graph is replayed.
cudaError_t record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return cudaGetLastError();
  if (st == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  return cudaEventRecord(e, s);
}

// Validation of a call; on success every member is well formed and aligned.
// ldy / col0 (either may be null: N and 0) give each member's output window.
int validate_call(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                  const int64_t* ldy, const int* col0) {
  if (count < 1 || count > 3) return fail(TFX_EINVAL, "group count %d outside 1..3", count);
  if (rows < 0) return fail(TFX_EINVAL, "rows=%d", rows);
  if (!x || !ys) return fail(TFX_EINVAL, "null x or ys");
  for (int i = 0; i < count; i++) {
    int rc = validate(ws[i]);
    if (rc) return rc;
    if (!ys[i]) return fail(TFX_EINVAL, "null y of member %d", i);
    if (!aligned16(ys[i])) return fail(TFX_EALIGN, "y of member %d is not 16-byte aligned", i);
    if (ws[i]->K != ws[0]->K || ws[i]->bits != ws[0]->bits || ws[i]->act != ws[0]->act)
      return fail(TFX_EUNSUPPORTED, "group members must share K, bits and act");
    const int c0 = col0 ? col0[i] : 0;
    const long long ld = ldy ? ldy[i] : ws[i]->N;
    if (c0 < 0 || c0 >= ws[i]->N || c0 % 8)
      return fail(TFX_EINVAL, "col0=%d of member %d: a multiple of 8 in [0, N=%d)", c0, i, ws[i]->N);
    if (ld < ws[i]->N - c0 || ld % 8)
      return fail(TFX_EINVAL, "ldy=%lld of member %d: a multiple of 8 and at least N - col0 = %d", ld, i,
                  ws[i]->N - c0);
  }
  if (!aligned16(x)) return fail(TFX_EALIGN, "x is not 16-byte aligned");
  return 0;
}

int run(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[], const int64_t* ldy,
        const int* col0, cudaStream_t s) {
  int rc = validate_call(ws, count, x, rows, ys, ldy, col0);
  if (rc) return rc;
  if (rows == 0) return 0;
  tfx::Scratch sc = {};
  for (int i = 0; i < count; i++) {
    Priv* pv = static_cast<Priv*>(ws[i]->priv);
    if (!pv || pv->max_rows < rows)
      return fail(TFX_ENOTRESERVED, "member %d reserved for %d rows, called with %d", i, pv ? pv->max_rows : 0,
                  rows);
    sc.xf[i] = pv->xf;
    sc.partial[i] = pv->partial;
    sc.counters[i] = pv->counters + tfx::kErrorInts;
    if (i == 0) {
      sc.err = pv->counters;
      sc.lev = pv->lev;
    }
  }
  return tfx::launch_layer(ws, count, x, rows, ys, ldy, col0, s, sc, g_pdl.load(std::memory_order_relaxed));
}

int grow(void** p, size_t* have, size_t want, cudaStream_t s, Priv* pv, bool zero) {
  if (want <= *have) return 0;
  void* np = nullptr;
  const tfx_exl3_driver d = drv();
  if (d.alloc(&np, want, s) != 0 || !np) return fail(TFX_ECUDA, "allocation of %zu bytes failed", want);
  pv->allocs++;
  if (zero) {
    if (d.memset0(np, want, s) != 0) return fail(TFX_ECUDA, "zeroing %zu bytes failed", want);
    pv->memsets++;
  }
  if (*p) d.free(*p, s);
  *p = np;
  *have = want;
  return 0;
}

}  // namespace

namespace tfx {

int chunks_of(int K) {
  const int TK = K / 16;
  int c = 1;
  while (c < kMaxChunks && 2 * c <= TK / 4) c *= 2;
  return c;
}

// Rows of rotated x a call lays out: the decode-rows kernels read whole row
// tiles of 8*NR rows (16, 16, 32, 64), the tensor-core kernel 16-row groups;
// the rows past `rows` are written as zeros.
int x_rows_padded(int rows) {
  const int r16 = (rows + 15) / 16 * 16;
  if (rows > kRowsMaxRows) return r16;
  return rows <= 16 ? 16 : rows <= 32 ? 32 : 64;
}

size_t xf_bytes_needed(const tfx_exl3_weight* w, int rows) { return (size_t)x_rows_padded(rows) * w->K * 2; }

size_t partial_bytes_needed(const tfx_exl3_weight* w, int rows) {
  const int C = chunks_of(w->K), TN = w->N / 16;
  // decode-rows slabs: at most 16 rows with a grouping that depends on TN, or
  // up to kRowsMaxRows rows at one chunk per warp
  const int small = rows < 16 ? rows : 16;
  size_t need = (size_t)(C / (rows_gw(C) * rows_group(TN, C, small))) * small * w->N * 4;
  if (rows > 16) {
    const int mid = rows < kRowsMaxRows ? rows : kRowsMaxRows;
    const size_t m = (size_t)(C / rows_gw(C)) * mid * w->N * 4;
    need = m > need ? m : need;
  }
  // tensor-core slabs: up to kTcRowsMax rows, one pass of at most C/2 slabs
  // (a unit holds at least one chunk pair); above that one slab per pass
  // (each unit holds all C chunks), i.e. every row's z once; a weight reserved
  // for more rows also serves the shorter calls
  const int rp = rows < kTcRowsMax ? rows : kTcRowsMax;
  size_t tc = (size_t)(C / 2) * rp * w->N * 4;
  // decode-rows folds through global slabs: one slab per chunk, every row the
  // decode-rows kernel serves
  const size_t fg = (size_t)C * (rows < kRowsMaxRows ? rows : kRowsMaxRows) * w->N * 4;
  if (fg > tc) tc = fg;
  const size_t whole = (size_t)((rows + kTcRowsNoSpill - 1) / kTcRowsNoSpill) * kTcRowsNoSpill * w->N * 4;
  if (whole > tc) tc = whole;
  return tc > need ? tc : need;
}

size_t counter_bytes_needed(const tfx_exl3_weight* w, int rows) {
  // the most passes any call of up to `rows` rows may use (64-row passes)
  return (size_t)(kErrorInts + tc_passes(rows, false) * (w->N / 128)) * sizeof(int);
}

size_t level_bytes_needed(int rows) {
  // a tensor-core call parks chunk-tree levels in global scratch only when its
  // TMEM regions are wider than 64 columns (more than 64 rows per pass): up to
  // 64, TMEM holds all three levels above the pairs next to the four regions
  if (rows <= 64) return 0;
  return (size_t)sm_count() * kTcSpillLevels * kTcRowsMax * 128 * sizeof(float);
}

int launch_layer(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                 const int64_t* ldy, const int* col0, cudaStream_t s, const Scratch& sc, int pdl) {
  const int K = ws[0]->K, bits = ws[0]->bits;

  // rotation of x, once for all members
  RotArgs ra = {};
  ra.x = x;
  ra.count = count;
  ra.rows = rows;
  ra.rows_pad = (rows + 15) / 16 * 16;
  long long weights = 0;
  for (int i = 0; i < count; i++) weights += (long long)K * ws[i]->N;
  const Family f = pick(bits, rows);
  if (f.rows()) ra.rows_pad = tfx::x_rows_padded(rows);  // whole row tiles, zero-padded
  ra.K = K;
  ra.act = ws[0]->act;
  for (int i = 0; i < count; i++) {
    ra.suh[i] = reinterpret_cast<const __half*>(ws[i]->suh);
    ra.xf[i] = sc.xf[i];
  }
  ra.layout = f.rows() ? 0 : 1;
  const bool spill = sc.lev != nullptr;
  ra.rp_tc = tc_rows_per_pass(rows, spill);  // 128 for every call the clustered kernel serves
  const long long items = (long long)ra.rows_pad * (K / 128);
  int rc = 0;

  // one grid over every member's CTAs
  LinearArgs la = {};
  la.count = count;
  la.K = K;
  la.TK = K / 16;
  la.rows = rows;
  const int per_pass = f.kind == kTensor ? tc_rows_per_pass(rows, spill) : kRowsPerPass;
  la.passes = (rows + per_pass - 1) / per_pass;
  la.rp = rows < per_pass ? rows : per_pass;
  la.act = ws[0]->act;
  la.err = sc.err;
  la.spin = g_spin.load(std::memory_order_relaxed);
  long long ctas = 0;
  int tcG = 0;
  long long all_blocks = 0;
  for (int i = 0; i < count; i++) all_blocks += ws[i]->N / 128;
  const int fold_mode = f.kind == kRowsWarp ? fold_mode_for(rows, all_blocks) : tfx::kFoldCluster;
  const bool fold_slabs = fold_mode != tfx::kFoldCluster;  // no clusters: chunk sums in global slabs
  if (f.kind == kTensor) {
    long long blocks = 0;
    for (int i = 0; i < count; i++) blocks += ws[i]->N / 128;
    tcG = tc_group(blocks, rows, chunks_of(K), K / 16, sm_count(), spill);
  }
  for (int i = 0; i < count; i++) {
    const tfx_exl3_weight* w = ws[i];
    Member& m = la.m[i];
    m.trellis = w->trellis;
    m.stride = w->tile_row_stride;
    m.svh = reinterpret_cast<const __half*>(w->svh);
    m.suh = reinterpret_cast<const __half*>(w->suh);
    m.xf = sc.xf[i];
    m.y = ys[i];
    m.ldy = ldy ? ldy[i] : w->N;
    m.col0 = col0 ? col0[i] : 0;
    m.partial = sc.partial[i];
    m.counters = sc.counters[i];
    m.N = w->N;
    m.NB = w->N / 128;
    m.C = chunks_of(K);
    m.cta_begin = (int)ctas;
    if (f.kind == kRowsWarp) {
      // one CTA per (128-column block, chunk); the C CTAs of a block are one
      // cluster that folds the chunk sums in distributed shared memory
      m.G = 1;
      m.TC = f.ncol;
      m.P = fold_slabs ? m.C : 1;  // slabs of a block: one per chunk when folded through slabs
      m.arrivals = fold_mode == tfx::kFoldCounter ? m.C : 0;
      ctas += (long long)m.NB * m.C;
    } else if (f.kind == kRowsCta) {
      const int TN = w->N / 16;
      m.G = rows_group(TN, m.C, rows);
      m.TC = rows_gw(m.C);  // the decode-rows kernel reads its warp-group count here
      m.P = m.C / (m.TC * m.G);
      m.arrivals = (8 / kRowsTC) * m.P;
      ctas += (long long)(TN / kRowsTC) * m.P;
    } else {
      // work units (pass, block, chunk group); cta_begin holds the member's first unit
      m.G = tcG;
      m.TC = 8;
      m.P = m.C / m.G;
      m.arrivals = m.P;
      ctas += (long long)m.NB * m.P * la.passes;
    }
    m.log2G = __builtin_ctz(m.G);
  }
  la.items = ctas;
  if (ctas > 0x7fffffffLL) return fail(TFX_EUNSUPPORTED, "grid of %lld CTAs", ctas);
  size_t smem = f.kind == kTensor ? kTcDynSmem : 0;
  if (f.kind == kTensor) {
    // the members' trellis words as 2-D tensors, boxes of 4 tiles x 4 tile rows
    for (int i = 0; i < count; i++) {
      rc = encode_trellis_map(ws[i], tfx::tc_word_box_words(bits), tfx::kTcBoxRows, &la.tm[i]);
      if (rc) return rc;
    }
  }
  if (f.kind == kRowsWarp) {
    // tensor maps of the members' trellis words and the box shape
    long long clusters = 0;
    for (int i = 0; i < count; i++) clusters += ws[i]->N / 128;
    const WarpStaging stg = warp_staging(K, bits, f.ncol, f.nr, clusters);
    la.box_rows = stg.H;
    la.ring_boxes = stg.R;
    la.x_rows = stg.XH;
    la.x_whole = stg.x_whole;
    // up to kFuseRotRows rows, on calls of fewer than kFuseRotWeights weights,
    // each CTA rotates its chunk of x itself: a few warp-items per CTA, cheaper
    // than the rotation kernel and its launch on the critical path of a
    // latency-bound call (measured on GB300: 5120 x 5120 at 1 row 13.9 -> 12.8
    // us); on large calls the redundant rotation costs more than it saves
    // (LM head at 1 row 444 -> 482 us)
    la.fuse_rot = (rows <= kFuseRotRows && stg.x_whole && weights < kFuseRotWeights) ? 1 : 0;
    // CTAs leave the closing cluster barrier early only where other clusters
    // wait for their SM slots (about 54-68 clusters of 16 CTAs are resident
    // at once on 152 SMs)
    la.early_arrive = clusters > kEarlyArriveClusters ? 1 : 0;
    la.fold_mode = fold_mode;
    la.x = x;
    for (int i = 0; i < count; i++) {
      rc = encode_trellis_map(ws[i], f.ncol * 8 * bits, stg.H, &la.tm[i]);
      if (rc) return rc;
    }
    smem = (size_t)tfx::warp_smem_bytes(stg.H, stg.R, stg.XH, stg.x_whole, bits, f.ncol, f.nr, rows);
    // the largest carveout, set once: both operands come through shared memory;
    // clusters of 16 CTAs (16 chunks) need the non-portable size opt-in
    rc = set_carveout(f.fn, 100);
    if (rc) return rc;
    rc = allow_big_clusters(f.fn);
    if (rc) return rc;
  }
  rc = set_smem(f.fn, smem);
  if (rc) return rc;
  TcArgs ta;
  ta.la = la;
  ta.units = (int)ctas;
  ta.RP = per_pass;
  ta.NMf = per_pass < ra.rows_pad ? per_pass : ra.rows_pad;
  ta.tlev = tc_tmem_levels(ta.NMf);
  ta.err = sc.err;
  ta.lev = sc.lev;
  if (f.kind == kTensor && __builtin_ctz(tcG) - 1 > ta.tlev && !sc.lev)
    return fail(TFX_EUNSUPPORTED, "tensor-core launch needs chunk-tree level scratch");
  if (f.kind == kTensor) {
    const long long S = sm_count();
    ctas = ctas < S ? ctas : S;  // persistent: one CTA per SM at most
  }
  // programmatic dependent launch per kernel (see env_pdl): in the automatic
  // mode only a decode-rows call with its own rotation launch takes it, on
  // both of its launches
  const bool pdl_auto = pdl == 2 && f.kind == kRowsWarp && !la.fuse_rot;
  const bool pdl_rot = pdl == 1 || pdl_auto, pdl_lin = pdl == 1 || pdl_auto;
  const bool pdl_comb = pdl == 1 || (pdl == 2 && fold_mode == tfx::kFoldCombine);
  // everything that can fail on the host is done: enqueue the rotation, then the linear kernel
  if (!la.fuse_rot) {
    rc = launch(reinterpret_cast<const void*>(&rot_kernel), dim3((unsigned)((items + 7) / 8)), dim3(256), 0, s, &ra,
                pdl_rot);
    if (rc) return rc;
  }
  cudaEvent_t eb = g_ev_before, ea = g_ev_after;
  g_ev_before = g_ev_after = nullptr;
  if (eb && record_event(eb, s) != cudaSuccess) return fail(TFX_ECUDA, "cudaEventRecord");
  const int cluster = f.kind == kRowsWarp && !fold_slabs ? chunks_of(K) : 1;
  rc = f.kind != kTensor ? launch(f.fn, dim3((unsigned)ctas), dim3(f.wpc * 32), smem, s, &la, pdl_lin, cluster)
                         : launch(f.fn, dim3((unsigned)ctas), dim3(f.wpc * 32), smem, s, &ta, pdl_lin);
  if (rc) return rc;
  if (f.kind == kTensor || fold_mode == tfx::kFoldCombine) {
    // fold every block's slabs (one, when a unit covered all C chunks), rotate
    // back and store y: one warp per (row, block)
    CombineArgs ca = {};
    ca.la = la;
    ca.RP = per_pass;
    long long warps = 0;
    for (int i = 0; i < count; i++) {
      ca.items[i] = (long long)rows * la.m[i].NB;
      warps += ca.items[i];
    }
    if (warps > 0) {
      rc = launch(reinterpret_cast<const void*>(&tc_combine_kernel), dim3((unsigned)((warps + 7) / 8)), dim3(256), 0,
                  s, &ca, pdl_comb);
      if (rc) return rc;
    }
  }
  if (ea && record_event(ea, s) != cudaSuccess) return fail(TFX_ECUDA, "cudaEventRecord");
  return 0;
}

}  // namespace tfx

extern "C" {

int tfx_exl3_linear(tfx_exl3_weight* w, const void* x, int rows, void* y, cudaStream_t stream) {
  tfx_exl3_weight* ws[1] = {w};
  void* ys[1] = {y};
  return run(ws, 1, x, rows, ys, nullptr, nullptr, stream);
}

int tfx_exl3_group(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                   cudaStream_t stream) {
  if (!ws) return fail(TFX_EINVAL, "null member list");
  return run(ws, count, x, rows, ys, nullptr, nullptr, stream);
}

int tfx_exl3_group_into(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                        const int64_t ldy[], const int col0[], cudaStream_t stream) {
  if (!ws) return fail(TFX_EINVAL, "null member list");
  if (!ldy || !col0) return fail(TFX_EINVAL, "null ldy or col0");
  return run(ws, count, x, rows, ys, ldy, col0, stream);
}

int tfx_exl3_chain(const tfx_exl3_step* steps, int nsteps, int rows, int pdl, cudaStream_t stream) {
  if (!steps || nsteps < 1) return fail(TFX_EINVAL, "chain of %d steps", nsteps);
  if (pdl < 0 || pdl > 2) return fail(TFX_EINVAL, "chain pdl mode %d (0, 1 or 2)", pdl);
  // every step is validated (shapes, alignment, reserve) before anything is enqueued
  for (int i = 0; i < nsteps; i++) {
    const tfx_exl3_step& st = steps[i];
    if (!st.ws) return fail(TFX_EINVAL, "step %d: null member list", i);
    int rc = validate_call(st.ws, st.count, st.x, rows, st.ys, nullptr, nullptr);
    if (rc) return fail(rc, "step %d: %s", i, g_err.c_str());
    for (int m = 0; m < st.count; m++) {
      const Priv* pv = static_cast<const Priv*>(st.ws[m]->priv);
      if (!pv || pv->max_rows < rows)
        return fail(TFX_ENOTRESERVED, "step %d member %d reserved for %d rows, chain of %d", i, m,
                    pv ? pv->max_rows : 0, rows);
    }
  }
  if (rows == 0) return 0;
  for (int i = 0; i < nsteps; i++) {
    const tfx_exl3_step& st = steps[i];
    tfx::Scratch sc = {};
    for (int m = 0; m < st.count; m++) {
      Priv* pv = static_cast<Priv*>(st.ws[m]->priv);
      sc.xf[m] = pv->xf;
      sc.partial[m] = pv->partial;
      sc.counters[m] = pv->counters + tfx::kErrorInts;
      if (m == 0) {
        sc.err = pv->counters;
        sc.lev = pv->lev;
      }
    }
    const int rc = tfx::launch_layer(st.ws, st.count, st.x, rows, st.ys, nullptr, nullptr, stream, sc, pdl);
    if (rc) return fail(rc, "step %d: %s", i, g_err.c_str());
  }
  return 0;
}

int tfx_exl3_columns(const tfx_exl3_weight* w, int from, int n, tfx_exl3_weight* view_out) {
  int rc = validate(w);
  if (rc) return rc;
  if (!view_out) return fail(TFX_EINVAL, "null view_out");
  if (from < 0 || n <= 0 || from % 128 || n % 128 || (long long)from + n > w->N)
    return fail(TFX_EINVAL, "columns(from=%d, n=%d) is not a whole-block range of N=%d", from, n, w->N);
  tfx_exl3_weight v = *w;
  v.trellis = w->trellis + (long long)(from / 16) * 8 * w->bits;
  v.svh = w->svh + from;
  v.N = n;
  v.priv = nullptr;
  *view_out = v;
  return 0;
}

int tfx_exl3_reserve(tfx_exl3_weight* w, int max_rows, cudaStream_t stream) {
  int rc = validate(w);
  if (rc) return rc;
  if (max_rows < 1) return fail(TFX_EINVAL, "max_rows=%d", max_rows);
  Priv* pv = static_cast<Priv*>(w->priv);
  if (!pv) {
    pv = new Priv();
    w->priv = pv;
  }
  if (max_rows <= pv->max_rows) return 0;
  rc = grow(reinterpret_cast<void**>(&pv->xf), &pv->xf_bytes, tfx::xf_bytes_needed(w, max_rows), stream, pv, false);
  if (!rc)
    rc = grow(reinterpret_cast<void**>(&pv->partial), &pv->partial_bytes, tfx::partial_bytes_needed(w, max_rows),
              stream, pv, false);
  if (!rc)
    rc = grow(reinterpret_cast<void**>(&pv->counters), &pv->counter_bytes, tfx::counter_bytes_needed(w, max_rows),
              stream, pv, true);
  if (!rc && tfx::level_bytes_needed(max_rows))
    rc = grow(reinterpret_cast<void**>(&pv->lev), &pv->lev_bytes, tfx::level_bytes_needed(max_rows), stream, pv, false);
  if (rc) return rc;
  pv->max_rows = max_rows;
  return 0;
}

int tfx_exl3_release(tfx_exl3_weight* w) {
  if (!w) return fail(TFX_EINVAL, "null weight");
  Priv* pv = static_cast<Priv*>(w->priv);
  if (!pv) return 0;
  const tfx_exl3_driver d = drv();
  if (d.alloc == rt_alloc) cudaDeviceSynchronize();
  if (pv->xf) d.free(pv->xf, nullptr);
  if (pv->partial) d.free(pv->partial, nullptr);
  if (pv->counters) d.free(pv->counters, nullptr);
  if (pv->lev) d.free(pv->lev, nullptr);
  if (d.alloc == rt_alloc) cudaDeviceSynchronize();
  delete pv;
  w->priv = nullptr;
  return 0;
}

int tfx_exl3_reset_counters(tfx_exl3_weight* w, cudaStream_t stream) {
  if (!w) return fail(TFX_EINVAL, "null weight");
  Priv* pv = static_cast<Priv*>(w->priv);
  if (!pv || !pv->counters) return fail(TFX_ENOTRESERVED, "weight not reserved");
  if (drv().memset0(pv->counters, pv->counter_bytes, stream) != 0) return fail(TFX_ECUDA, "zeroing counters");
  pv->memsets++;
  return 0;
}

int tfx_exl3_debug_decode(const tfx_exl3_weight* w, uint16_t* W_out, cudaStream_t stream) {
  int rc = validate(w);
  if (rc) return rc;
  if (!W_out) return fail(TFX_EINVAL, "null W_out");
  tfx::DecodeArgs da;
  da.trellis = w->trellis;
  da.stride = w->tile_row_stride;
  da.W = reinterpret_cast<__half*>(W_out);
  da.K = w->K;
  da.N = w->N;
  const long long tiles = (long long)(w->K / 16) * (w->N / 16);
  return launch(kernels(w->bits).decode, dim3((unsigned)((tiles + 7) / 8)), dim3(256), 0, stream, &da, false);
}

int tfx_exl3_debug_launch_shape(int K, int bits, int rows, int64_t blocks, int sm_count_, int* family,
                                int* chunks_per_unit) {
  if (K <= 0 || K % 128 || bits < 1 || bits > 8 || rows < 1 || blocks < 1 || sm_count_ < 0 || !family ||
      !chunks_per_unit)
    return fail(TFX_EINVAL, "debug_launch_shape: K a positive multiple of 128, bits 1..8, rows >= 1, "
                            "blocks >= 1, sm_count >= 0, non-null outputs");
  const Family f = pick(bits, rows);
  *family = (int)f.kind;
  *chunks_per_unit = f.kind == kTensor ? tc_group(blocks, rows, tfx::chunks_of(K), K / 16,
                                                  sm_count_ ? sm_count_ : sm_count(), true)
                                         : 0;
  return 0;
}

int tfx_exl3_plan(const tfx_exl3_weight* w, int* chunks, int* tiles_per_chunk) {
  int rc = validate(w);
  if (rc) return rc;
  const int C = tfx::chunks_of(w->K);
  if (chunks) *chunks = C;
  if (tiles_per_chunk) *tiles_per_chunk = (w->K / 16) / C;
  return 0;
}

int tfx_exl3_stats(const tfx_exl3_weight* w, int64_t* allocs, int64_t* memsets) {
  if (!w) return fail(TFX_EINVAL, "null weight");
  const Priv* pv = static_cast<const Priv*>(w->priv);
  if (allocs) *allocs = pv ? pv->allocs : 0;
  if (memsets) *memsets = pv ? pv->memsets : 0;
  return 0;
}

int tfx_exl3_set_variant(int variant) {
  if (variant < 0 || variant > 4) return g_variant.load();
  return g_variant.exchange(variant);
}

int64_t tfx_exl3_debug_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int tfx_exl3_set_pdl(int mode) {
  if (mode < 0 || mode > 2) return fail(TFX_EINVAL, "pdl mode %d (0, 1 or 2)", mode);
  return g_pdl.exchange(mode);
}

int64_t tfx_exl3_debug_set_spin_limit(int64_t clocks) {
  return g_spin.exchange(clocks > 0 ? clocks : tfx::kSpinClocks);
}

int tfx_exl3_debug_set_driver(const tfx_exl3_driver* d) {
  std::lock_guard<std::mutex> lk(g_drv_mu);
  if (!d) {
    g_drv_hooks = tfx_exl3_driver{rt_alloc, rt_free, rt_memset0};
    return 0;
  }
  if (!d->alloc || !d->free || !d->memset0) return fail(TFX_EINVAL, "driver hooks must all be set");
  g_drv_hooks = *d;
  return 0;
}

int tfx_exl3_debug_decode_rate(int bits, int tiles_per_warp, float* sink, int* sink_floats, int64_t* weights,
                               cudaStream_t stream) {
  if (bits < 1 || bits > 8 || tiles_per_warp < 1 || !sink_floats || !weights)
    return fail(TFX_EINVAL, "debug_decode_rate: bits 1..8, tiles_per_warp >= 1, non-null sink_floats and weights");
  const int ctas = sm_count() * tfx::kRateCtasPerSm;
  *sink_floats = ctas * tfx::kRateWarps;
  *weights = (int64_t)ctas * tfx::kRateWarps * tiles_per_warp * 256;
  if (!sink) return 0;
  if (!aligned16(sink)) return fail(TFX_EALIGN, "sink must be 16-byte aligned");
  tfx::RateArgs ra{tiles_per_warp, sink};
  return launch(kernels(bits).decode_rate, dim3((unsigned)ctas), dim3(tfx::kRateWarps * 32), 0, stream, &ra, false);
}

int tfx_exl3_debug_error(const tfx_exl3_weight* w, int* device_error) {
  if (!w || !device_error) return fail(TFX_EINVAL, "null argument");
  const Priv* pv = static_cast<const Priv*>(w->priv);
  if (!pv || !pv->counters) return fail(TFX_ENOTRESERVED, "weight not reserved");
  cudaError_t e = cudaMemcpy(device_error, pv->counters, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  return 0;
}

int tfx_exl3_debug_mark_events(cudaEvent_t before, cudaEvent_t after) {
  g_ev_before = before;
  g_ev_after = after;
  return 0;
}

const char* tfx_exl3_last_error(void) { return g_err.c_str(); }

}  // extern "C"

// Error reporting for the other C-ABI translation units.
namespace tfx {
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace tfx
