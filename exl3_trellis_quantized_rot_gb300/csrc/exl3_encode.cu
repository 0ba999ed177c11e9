// Synthetic trellis encoder for sm_103a: grid targets -> trellis words.
//
// The pages quantize with trained checkpoints and never show their encoder;
// the decode rule is the build's bit-shift trellis (exl3_kernels.cuh). The
// encoder follows QTIP (Tseng et al., 2024, "QTIP: Quantization with
// Trellises and Incoherence Processing"): a Viterbi search over the
// shift-register trellis for the tail-biting code whose decoded values are
// closest, in summed squared error, to the targets, with QTIP's two-pass
// approximation of the tail-biting constraint. Per 16x16 tile:
//   * targets are integers on the value grid (units of 1/128), clamped to
//     [-1024, 1023], so every path cost is an exact integer below 2^30;
//   * state s (16 bits) moves to s' = (s >> bits) | (u << (16 - bits)); the
//     predecessors of s' are the group P = s' & m (m = 2^(16-bits) - 1) of
//     states (P << bits) | v, v < 2^bits;
//   * step j: best[P] = min over v of cost[(P << bits) | v] (ties: smaller
//     v), then cost'[s] = best[s & m] + (value(s) - T[j])^2 for every s;
//   * pass 1 runs on the targets rotated by 128 weights with any start and
//     end; its state at the tile's weight 0 gives the overlap bits c;
//   * pass 2 runs on the targets in order with starts (s & m) == c (others
//     cost 2^30) and ends (s >> bits) == c (smallest cost, then smallest
//     state), which closes the circular stream;
//   * the best path is traced back through the stored argmins; weight j's
//     `bits` stream bits are the low bits of its state.
// The same integer decisions as the CPU oracle, so the words are identical.
//
// Work layout: one CTA of 512 threads per tile at a time, as many CTAs per SM
// as fit (persistent over tiles): a tile is a chain of 510 dependent steps, so
// throughput grows with the tiles in flight. The two cost arrays (2^16 int32 each) and the argmins of every step
// (2^(16-bits) bytes) live in a per-CTA slice of caller scratch (L2-resident
// while the tile runs); best[] lives in shared memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tfx_exl3.h"
#include "exl3_internal.h"

namespace tfx {

// Threads per CTA: 1024 at 1 and 2 bits, where best[] (128 / 64 KB of shared
// memory) lets only one or two CTAs share an SM, 512 above, where three CTAs
// per SM (the register limit) keep more tiles in flight. Measured on GB300
// (1024 x 1024 targets, grid from occupancy): 512 threads at every width gave
// 7.9k / 10.8k tiles/s at 1 / 2 bits, this choice 15.1k / 15.9k; at 4 bits
// 512 threads give 10.4k against 9.8k for one 1024-thread CTA per SM.
__host__ __device__ constexpr int enc_threads(int bits) { return bits <= 2 ? 1024 : 512; }
constexpr uint32_t kEncInf = 1u << 30;

struct EncodeArgs {
  const int16_t* targets;  // K x N, row-major, grid units
  uint32_t* trellis;       // tile layout, tile row stride (N/16)*8*bits words
  long long* sq_err;       // per tile (or null)
  unsigned char* scratch;  // gridDim.x slices of enc_slice_bytes(bits)
  int K, N;
  long long tiles;
};

__host__ __device__ constexpr size_t enc_slice_bytes(int bits) {
  return (size_t)2 * 65536 * 4 + (size_t)256 * (65536 >> bits);
}
// Dynamic shared memory of the kernel: best[] per predecessor group.
__host__ __device__ constexpr size_t enc_smem_bytes(int bits) { return (size_t)(65536 >> bits) * 4; }

// The decode rule's integer value of a state: byte sum of the hashed state - 510.
__device__ __forceinline__ int enc_value(uint32_t s) {
  const uint32_t h = s * kHashMul + kHashAdd;
  return (int)__dp4a(h, 0x01010101u, 0u) - 510;
}

// One Viterbi pass over the 256 targets T (shared memory). constrain: starts
// with (s & m) == c, ends with (s >> BITS) == c. Leaves the argmins of steps
// 1..255 in dec and returns the best end state and cost in *end_s / *end_cost
// (block-uniform).
template <int BITS>
__device__ void enc_pass(const int* T, bool constrain, uint32_t c, uint32_t* cost, uint32_t* next,
                         unsigned char* dec, uint32_t* best, uint32_t* red_c, uint32_t* red_s,
                         uint32_t* end_s, uint32_t* end_cost) {
  constexpr int kEncThreads = enc_threads(BITS);
  constexpr int G = 1 << BITS;                 // predecessors per group
  constexpr uint32_t NP = 65536u >> BITS;      // groups
  constexpr uint32_t m = NP - 1u;
  constexpr int SEG = G < 32 ? G : 32;         // lanes per group in the min
  constexpr int PER = G / SEG;                 // elements per lane
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (uint32_t s = tid; s < 65536u; s += kEncThreads) {
    const int d = enc_value(s) - T[0];
    __stcg(cost + s, (!constrain || (s & m) == c) ? (uint32_t)(d * d) : kEncInf);
  }
  __syncthreads();
  for (int j = 1; j < 256; j++) {
    // best predecessor of each group: a segment of SEG lanes per group, each
    // lane the minimum of its PER elements, then a tree of shuffles that keeps
    // the smaller cost and, on a tie, the smaller v
    const int gpw = 32 / SEG;  // groups per warp iteration
    for (uint32_t P0 = (uint32_t)warp * gpw; P0 < NP; P0 += (kEncThreads / 32) * gpw) {
      const uint32_t P = P0 + lane / SEG;
      const int sl = lane % SEG;
      uint32_t bc = kEncInf * 2u, bv = 0;
      if (P < NP) {
#pragma unroll
        for (int i = 0; i < PER; i++) {
          const uint32_t v = (uint32_t)(sl + SEG * i);
          const uint32_t x = __ldcg(cost + (P << BITS) + v);
          if (x < bc) {
            bc = x;
            bv = v;
          }
        }
      }
#pragma unroll
      for (int o = 1; o < SEG; o <<= 1) {
        const uint32_t oc = __shfl_xor_sync(0xffffffffu, bc, o), ov = __shfl_xor_sync(0xffffffffu, bv, o);
        if (oc < bc || (oc == bc && ov < bv)) {
          bc = oc;
          bv = ov;
        }
      }
      if (sl == 0 && P < NP) {
        best[P] = bc;
        dec[(size_t)j * NP + P] = (unsigned char)bv;
      }
    }
    __syncthreads();
    for (uint32_t s = tid; s < 65536u; s += kEncThreads) {
      const int d = enc_value(s) - T[j];
      __stcg(next + s, best[s & m] + (uint32_t)(d * d));
    }
    __syncthreads();
    uint32_t* t = cost;
    cost = next;
    next = t;
  }
  // best end state: smallest cost, then smallest state
  uint32_t bc = 0xFFFFFFFFu, bs = 0xFFFFFFFFu;
  for (uint32_t s = tid; s < 65536u; s += kEncThreads) {
    if (constrain && (s >> BITS) != c) continue;
    const uint32_t x = __ldcg(cost + s);
    if (x < bc || (x == bc && s < bs)) {
      bc = x;
      bs = s;
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t oc = __shfl_xor_sync(0xffffffffu, bc, o), os = __shfl_xor_sync(0xffffffffu, bs, o);
    if (oc < bc || (oc == bc && os < bs)) {
      bc = oc;
      bs = os;
    }
  }
  if (lane == 0) {
    red_c[warp] = bc;
    red_s[warp] = bs;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t c0 = red_c[0], s0 = red_s[0];
    for (int w = 1; w < kEncThreads / 32; w++)
      if (red_c[w] < c0 || (red_c[w] == c0 && red_s[w] < s0)) {
        c0 = red_c[w];
        s0 = red_s[w];
      }
    *end_cost = c0;
    *end_s = s0;
  }
  __syncthreads();
}

template <int BITS>
__global__ void __launch_bounds__(enc_threads(BITS)) encode_kernel(const __grid_constant__ EncodeArgs a) {
  constexpr int kEncThreads = enc_threads(BITS);
  constexpr uint32_t NP = 65536u >> BITS;
  constexpr uint32_t m = NP - 1u;
  __shared__ int T[256], R[256];
  __shared__ uint32_t st[256];
  extern __shared__ __align__(16) unsigned char enc_dyn[];  // best[NP]
  uint32_t* best = reinterpret_cast<uint32_t*>(enc_dyn);
  __shared__ uint32_t red_c[kEncThreads / 32], red_s[kEncThreads / 32];
  __shared__ uint32_t end_s, end_cost;
  unsigned char* slice = a.scratch + (size_t)blockIdx.x * enc_slice_bytes(BITS);
  uint32_t* c0 = reinterpret_cast<uint32_t*>(slice);
  uint32_t* c1 = c0 + 65536;
  unsigned char* dec = slice + 2 * 65536 * 4;
  const int TN = a.N / 16;
  for (long long tile = blockIdx.x; tile < a.tiles; tile += gridDim.x) {
    const long long tk = tile / TN, tn = tile % TN;
    if (threadIdx.x < 256) {
      // weight j of the tile: the m16n8k16 A-fragment position of the decode rule
      const int j = threadIdx.x, lane = j >> 3, i = j & 7, g = lane >> 2, t = lane & 3;
      const int nl = g + 8 * ((i >> 1) & 1), kl = 2 * t + (i & 1) + 8 * (i >> 2);
      int v = a.targets[(16 * tk + kl) * (long long)a.N + 16 * tn + nl];
      v = v < -1024 ? -1024 : (v > 1023 ? 1023 : v);
      T[j] = v;
      R[(j + 128) & 255] = v;  // R[j'] = T[(j' + 128) % 256]
    }
    __syncthreads();
    // pass 1: rotated targets, any start and end; the state at rotated index 128
    enc_pass<BITS>(R, false, 0u, c0, c1, dec, best, red_c, red_s, &end_s, &end_cost);
    if (threadIdx.x == 0) {
      uint32_t s = end_s;
      for (int j = 255; j > 128; j--) s = ((s & m) << BITS) | __ldcg(dec + (size_t)j * NP + (s & m));
      st[0] = s & m;  // the overlap bits c
    }
    __syncthreads();
    const uint32_t c = st[0];
    __syncthreads();
    // pass 2: targets in order, the circle closed through c
    enc_pass<BITS>(T, true, c, c0, c1, dec, best, red_c, red_s, &end_s, &end_cost);
    if (threadIdx.x == 0) {
      uint32_t s = end_s;
      st[255] = s;
      for (int j = 255; j > 0; j--) {
        s = ((s & m) << BITS) | __ldcg(dec + (size_t)j * NP + (s & m));
        st[j - 1] = s;
      }
      if (a.sq_err) a.sq_err[tile] = (long long)end_cost;
    }
    __syncthreads();
    // pack: word w holds stream bits 32w .. 32w+31, weight j's bits at j*BITS
    if (threadIdx.x < 8 * BITS) {
      const int w = threadIdx.x;
      uint32_t word = 0;
      for (int bit = 0; bit < 32; bit++) {
        const int i = 32 * w + bit, j = i / BITS, t = i % BITS;
        word |= ((st[j] >> t) & 1u) << bit;
      }
      a.trellis[tk * (long long)TN * 8 * BITS + tn * 8 * BITS + w] = word;
    }
    __syncthreads();
  }
}

const void* encode_kernel_for(int bits) {
  switch (bits) {
    case 1: return reinterpret_cast<const void*>(&encode_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&encode_kernel<2>);
    case 3: return reinterpret_cast<const void*>(&encode_kernel<3>);
    case 4: return reinterpret_cast<const void*>(&encode_kernel<4>);
    case 5: return reinterpret_cast<const void*>(&encode_kernel<5>);
    case 6: return reinterpret_cast<const void*>(&encode_kernel<6>);
    case 7: return reinterpret_cast<const void*>(&encode_kernel<7>);
    default: return reinterpret_cast<const void*>(&encode_kernel<8>);
  }
}

}  // namespace tfx

namespace {

// Tiles in flight: every CTA the SMs hold at once (occupancy of the bit
// width's kernel), at most one per tile, at most max_ctas when given.
int enc_ctas(long long tiles, int bits, int max_ctas) {
  int sms = 0, dev = 0, per_sm = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    sms = 152;
  }
  const void* fn = tfx::encode_kernel_for(bits);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tfx::enc_smem_bytes(bits)) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, tfx::enc_threads(bits), tfx::enc_smem_bytes(bits)) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  long long c = (long long)sms * per_sm;
  if (tiles < c) c = tiles;
  if (max_ctas > 0 && c > max_ctas) c = max_ctas;
  return (int)(c < 1 ? 1 : c);
}

}  // namespace

extern "C" {

int tfx_exl3_encode_scratch_bytes(int K, int N, int bits, int max_ctas, size_t* bytes) {
  if (K <= 0 || N <= 0 || K % 16 || N % 16 || bits < 1 || bits > 8 || !bytes)
    return tfx::report_error(TFX_EINVAL, "encode_scratch_bytes: K, N positive multiples of 16, bits 1..8, bytes");
  const long long tiles = (long long)(K / 16) * (N / 16);
  *bytes = (size_t)enc_ctas(tiles, bits, max_ctas) * tfx::enc_slice_bytes(bits);
  return 0;
}

int tfx_exl3_encode(const int16_t* targets, int K, int N, int bits, uint32_t* trellis, int64_t* sq_err, void* scratch,
                    size_t scratch_bytes, int max_ctas, cudaStream_t stream) {
  if (K <= 0 || N <= 0 || K % 16 || N % 16 || bits < 1 || bits > 8)
    return tfx::report_error(TFX_EINVAL, "encode: K, N positive multiples of 16, bits 1..8");
  if (!targets || !trellis || !scratch) return tfx::report_error(TFX_EINVAL, "encode: null targets, trellis or scratch");
  if ((reinterpret_cast<uintptr_t>(scratch) | reinterpret_cast<uintptr_t>(trellis)) & 15u)
    return tfx::report_error(TFX_EALIGN, "encode: trellis and scratch must be 16-byte aligned");
  const long long tiles = (long long)(K / 16) * (N / 16);
  const int ctas = enc_ctas(tiles, bits, max_ctas);
  if (scratch_bytes < (size_t)ctas * tfx::enc_slice_bytes(bits))
    return tfx::report_error(TFX_EINVAL, "encode: scratch smaller than tfx_exl3_encode_scratch_bytes");
  tfx::EncodeArgs a;
  a.targets = targets;
  a.trellis = trellis;
  a.sq_err = reinterpret_cast<long long*>(sq_err);
  a.scratch = static_cast<unsigned char*>(scratch);
  a.K = K;
  a.N = N;
  a.tiles = tiles;
  void* args[1] = {&a};
  const void* fn = tfx::encode_kernel_for(bits);
  const size_t smem = tfx::enc_smem_bytes(bits);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  e = cudaLaunchKernel(fn, dim3((unsigned)ctas), dim3(tfx::enc_threads(bits)), args, smem, stream);
  if (e != cudaSuccess) return tfx::report_error(TFX_ECUDA, cudaGetErrorString(e));
  return 0;
}

}  // extern "C"
