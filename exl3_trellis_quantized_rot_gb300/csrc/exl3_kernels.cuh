// Device code of the EXL3 trellis linear for sm_103a.
//
// Decode rule (the build's own QTIP-style rule; the pages name the codebook
// "mul1" but do not define it — TensorFold PR #1467, section "Receipt",
// "synthetic weights at every 27B shape, mul1 4-bit"):
//   * a 16x16 tile is 8*BITS uint32 words = a circular stream of 256*BITS bits,
//     bit i = (word[i/32] >> (i%32)) & 1;
//   * weight j (0..255) has the 16-bit state of stream bits j*BITS .. j*BITS+15
//     (taken circularly), the first of them as the state's bit 0;
//   * h = state * 0x9E3779B1 + 0x7F4A7C15 (mod 2^32), v = sum of the 4 bytes of h,
//     value = (v - 510) / 128 — exact in FP16.
//   On the GPU: v + 0x6400 comes out of one dp4a (the FP16 bit pattern of 1024+v),
//   two such are packed into a half2 and one HFMA2 gives (1024+v)/128 - 1534/128,
//   a single rounding of an exactly representable result.
// Tile layout: weight j = 8*lane + i of a tile is the element the m16n8k16
//   A-operand register fragment gives lane `lane`, slot i, with the weights'
//   output column n as the fragment row and k as the fragment column:
//   n_local = g + 8*((i>>1)&1), k_local = 2t + (i&1) + 8*(i>>2), g = lane>>2,
//   t = lane&3. Tile (tk, tn) starts at word tk*stride + tn*8*BITS.
// Summation order (identical in every kernel variant, a function of K and the
//   plan only): K is cut into S splits and each split into Wk slices of whole
//   16-row tiles (contiguous, floor-divided). A slice is one chain of
//   m16n8k16 MMAs from zero in increasing k. A split's partial is the FP32
//   left fold of its slices in slice order; z is the left fold of the split
//   partials in split order (PR #1467, "The arithmetic" and the maintainers'
//   review: K ranges per warp, warp-order sums, split-order partials).
// Split-K combine: each CTA writes its split partial to scratch, fences and
//   increments the 128-column block's counter; the CTA that sees the last
//   arrival folds the partials in split order, applies the output rotation
//   and resets the counter to 0 (PR #1475, "What this changes": the last
//   arriving program resets counters[pass*NB + nb]). No CTA ever waits.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tfx {

constexpr uint32_t kHashMul = 0x9E3779B1u;
constexpr uint32_t kHashAdd = 0x7F4A7C15u;
constexpr float kInvSqrt128 = 0.08838834764831845f;  // 1/sqrt(128) rounded to FP32
constexpr int kRowsPerPass = 128;

struct Member {
  const uint32_t* trellis;  // first tile of this weight (or view)
  long long stride;         // uint32 words between tile rows
  const __half* svh;        // N
  const __half* xr;         // rotated x, rows x K, FP16
  void* y;                  // rows x N, act dtype
  float* partial;           // [pass][S][rp][N] FP32
  int* counters;            // [pass][NB]
  int N, NB, S, Wk;         // plan
  int TC;                   // 16-column tiles per CTA (= warps per CTA / Wk)
  int subs;                 // CTAs per 128-column block per split (= 8 / TC)
  int cta_begin;            // first blockIdx.x of this member
};

struct LinearArgs {
  Member m[3];
  int count;
  int K, TK;    // K and K/16
  int rows;     // total rows
  int passes;   // ceil(rows / 128)
  int rp;       // row stride of a partial slab = min(rows, 128)
  int act;      // 0 FP16, 1 BF16
};

struct RotArgs {
  const void* x;        // rows x K, act dtype
  const __half* suh[3]; // per member
  __half* xr[3];        // per member output
  int count, rows, K, act;
};

struct DecodeArgs {
  const uint32_t* trellis;
  long long stride;
  __half* W;  // K x N
  int K, N;
};

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Unnormalised 128-point Walsh-Hadamard transform (Sylvester order) of the
// 128 values a warp holds, 4 per lane (element 4*lane + e). Fixed butterfly
// order: strides 1, 2 in-thread, then 4..64 across lanes.
__device__ __forceinline__ void fwht128(float (&v)[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int m = 0; m < 5; m++) {
    const bool hi = (lane >> m) & 1;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      float o = __shfl_xor_sync(0xffffffffu, v[e], 1 << m);
      v[e] = hi ? (o - v[e]) : (v[e] + o);
    }
  }
}

// Words of one tile a lane needs: its 8 weights' windows span bits
// [8*lane*BITS, 8*lane*BITS + 7*BITS + 16), at most 2 words for BITS <= 4
// and 3 words above, counted from the word holding the first bit.
template <int BITS>
struct Geo {
  static constexpr int kWords = 8 * BITS;             // words per tile
  static constexpr int kRaw = BITS <= 4 ? 2 : 3;      // words loaded per lane
  static constexpr int kSpan = 7 * BITS + 16;         // bits used after alignment
  static constexpr int kNorm = (kSpan + 31) / 32;     // words after alignment
};

// Decode the lane's 8 weights from its (already bit-aligned) window into the
// 4 half2 registers of the m16n8k16 A fragment.
template <int BITS>
__device__ __forceinline__ void decode8(const uint32_t (&win)[Geo<BITS>::kNorm + 1], uint32_t (&a)[4]) {
  uint32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int p = i * BITS;
    const int q = p >> 5, sh = p & 31;
    uint32_t s = (sh == 0) ? win[q] : __funnelshift_r(win[q], win[q + 1], sh);
    s &= 0xFFFFu;
    const uint32_t h = s * kHashMul + kHashAdd;
    v[i] = __dp4a(h, 0x01010101u, 0x6400u);
  }
  const __half2 scale = __halves2half2(__ushort_as_half(0x2000), __ushort_as_half(0x2000));  // 2^-7
  const __half2 bias = __halves2half2(__float2half_rn(-1534.0f / 128.0f), __float2half_rn(-1534.0f / 128.0f));
#pragma unroll
  for (int m = 0; m < 4; m++) {
    uint32_t pk = __byte_perm(v[2 * m], v[2 * m + 1], 0x5410);
    __half2 hv = *reinterpret_cast<__half2*>(&pk);
    hv = __hfma2(hv, scale, bias);
    a[m] = *reinterpret_cast<uint32_t*>(&hv);
  }
}

// Load the raw words of the lane's window from a tile and align them so the
// lane's first weight starts at bit 0.
template <int BITS>
struct LaneWindow {
  int i0, i1, i2;  // word indices within the tile (circular)
  int off;         // bit offset of the first weight in word i0
  __device__ __forceinline__ void init(int lane) {
    const int P = 8 * lane * BITS;
    const int q0 = P >> 5;
    off = P & 31;
    i0 = q0;
    i1 = (q0 + 1) % Geo<BITS>::kWords;
    i2 = (q0 + 2) % Geo<BITS>::kWords;
  }
  __device__ __forceinline__ void load(const uint32_t* __restrict__ tile, uint32_t (&raw)[Geo<BITS>::kRaw]) const {
    raw[0] = __ldg(tile + i0);
    raw[1] = __ldg(tile + i1);
    if constexpr (Geo<BITS>::kRaw > 2) raw[2] = __ldg(tile + i2);
  }
  __device__ __forceinline__ void align(const uint32_t (&raw)[Geo<BITS>::kRaw],
                                        uint32_t (&win)[Geo<BITS>::kNorm + 1]) const {
    if constexpr ((8 * BITS) % 32 == 0) {
      // offsets are always 0 (BITS = 4, 8)
#pragma unroll
      for (int q = 0; q <= Geo<BITS>::kNorm; q++) win[q] = q < Geo<BITS>::kRaw ? raw[q] : 0u;
    } else {
#pragma unroll
      for (int q = 0; q <= Geo<BITS>::kNorm; q++) {
        uint32_t lo = q < Geo<BITS>::kRaw ? raw[q] : 0u;
        uint32_t hi = q + 1 < Geo<BITS>::kRaw ? raw[q + 1] : 0u;
        win[q] = __funnelshift_r(lo, hi, off);
      }
    }
  }
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The linear: one CTA = (128-column block nb, column sub-tile, split s, pass);
// warp (w, c) runs the chain of slice w over 16-column tile c of the CTA.
// NR = 8-row MMA groups per pass handled (rows of the pass <= 8*NR);
// WPC = warps per CTA; PF = tiles prefetched per warp.
template <int BITS, int NR, int WPC, int PF>
__global__ void __launch_bounds__(WPC * 32, (WPC <= 8 ? 4 : 1))
    linear_kernel(const __grid_constant__ LinearArgs a) {
  extern __shared__ float red[];  // [WPC][NR*8][16]
  __shared__ int s_last;
  griddep_wait();
  griddep_launch();

  int mi = 0;
  if (a.count > 1 && (int)blockIdx.x >= a.m[1].cta_begin) mi = 1;
  if (a.count > 2 && (int)blockIdx.x >= a.m[2].cta_begin) mi = 2;
  const Member& M = a.m[mi];

  int local = blockIdx.x - M.cta_begin;
  const int pass = local % a.passes;
  local /= a.passes;
  const int s = local % M.S;
  local /= M.S;
  const int nb = local / M.subs, sub = local % M.subs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int w = warp % M.Wk, c = warp / M.Wk;
  const int tn = nb * 8 + sub * M.TC + c;

  const int s0 = (s * a.TK) / M.S, s1 = ((s + 1) * a.TK) / M.S;
  const int t0 = s0 + (w * (s1 - s0)) / M.Wk, t1 = s0 + ((w + 1) * (s1 - s0)) / M.Wk;
  const int row0 = pass * kRowsPerPass;
  const int prow = min(kRowsPerPass, a.rows - row0);

  float acc[NR][4];
#pragma unroll
  for (int q = 0; q < NR; q++) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;

  if (c < M.TC) {
    LaneWindow<BITS> lw;
    lw.init(lane);
    const uint32_t* tp = M.trellis + (long long)t0 * M.stride + (long long)tn * (8 * BITS);
    // x fragment pointers: row 8q+g, columns 16*tk + 2t (+8)
    const uint32_t* xbase = reinterpret_cast<const uint32_t*>(M.xr + (long long)(row0 + g) * a.K + 16LL * t0 + 2 * t);
    const long long xq = 4LL * a.K;  // 8 rows, in uint32 units
    bool rv[NR];
#pragma unroll
    for (int q = 0; q < NR; q++) rv[q] = (8 * q + g) < prow;

    const int ntiles = t1 - t0;
    uint32_t ring[PF][Geo<BITS>::kRaw];
#pragma unroll
    for (int p = 0; p < PF; p++)
      if (p < ntiles) lw.load(tp + (long long)p * M.stride, ring[p]);

    for (int it = 0; it < ntiles; it += PF) {
#pragma unroll
      for (int p = 0; p < PF; p++) {
        const int tk = it + p;
        if (tk < ntiles) {
          uint32_t win[Geo<BITS>::kNorm + 1];
          lw.align(ring[p], win);
          if (tk + PF < ntiles) lw.load(tp + (long long)(tk + PF) * M.stride, ring[p]);
          uint32_t af[4];
          decode8<BITS>(win, af);
          const uint32_t* xp = xbase + 8LL * tk;
#pragma unroll
          for (int q = 0; q < NR; q++) {
            uint32_t b0 = 0u, b1 = 0u;
            if (rv[q]) {
              b0 = __ldg(xp + q * xq);
              b1 = __ldg(xp + q * xq + 4);
            }
            mma16816(acc[q], af, b0, b1);
          }
        }
      }
    }
  }

  // slice accumulators -> shared memory: red[warp][r][n_local]
  float* rw = red + warp * (NR * 8 * 16);
#pragma unroll
  for (int q = 0; q < NR; q++) {
    const int r0 = 8 * q + 2 * t;
    rw[r0 * 16 + g] = acc[q][0];
    rw[(r0 + 1) * 16 + g] = acc[q][1];
    rw[r0 * 16 + g + 8] = acc[q][2];
    rw[(r0 + 1) * 16 + g + 8] = acc[q][3];
  }
  __syncthreads();

  // fold slices in slice order, write this split's partial for the CTA's columns
  const int cols = M.TC * 16;
  const long long slab = (long long)(pass * M.S + s) * a.rp;
  float* part = M.partial;
  for (int idx = threadIdx.x; idx < prow * cols; idx += WPC * 32) {
    const int r = idx / cols, cc = idx - r * cols;
    const int cw = cc >> 4, nl = cc & 15;
    const float* src = red + (cw * M.Wk) * (NR * 8 * 16) + r * 16 + nl;
    float v = src[0];
    for (int ww = 1; ww < M.Wk; ww++) v += src[ww * (NR * 8 * 16)];
    part[(slab + r) * M.N + (long long)(nb * 8 + sub * M.TC) * 16 + cc] = v;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&M.counters[pass * M.NB + nb], 1);
    s_last = (old == M.S * M.subs - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last arrival: fold splits in split order, rotate back, scale by svh, store y
  const int n0 = nb * 128 + 4 * lane;
  float sv[4];
#pragma unroll
  for (int e = 0; e < 4; e++) sv[e] = __half2float(M.svh[n0 + e]);
  for (int r = warp; r < prow; r += WPC) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = __ldcg(part + ((long long)pass * M.S * a.rp + r) * M.N + n0 + e);
    for (int ss = 1; ss < M.S; ss++) {
#pragma unroll
      for (int e = 0; e < 4; e++) v[e] += __ldcg(part + ((long long)(pass * M.S + ss) * a.rp + r) * M.N + n0 + e);
    }
    fwht128(v, lane);
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = (v[e] * kInvSqrt128) * sv[e];
    const long long yo = (long long)(row0 + r) * M.N + n0;
    uint2 out;
    if (a.act == 0) {
      __half2 o0 = __floats2half2_rn(v[0], v[1]), o1 = __floats2half2_rn(v[2], v[3]);
      out.x = *reinterpret_cast<uint32_t*>(&o0);
      out.y = *reinterpret_cast<uint32_t*>(&o1);
      *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(M.y) + yo) = out;
    } else {
      __nv_bfloat162 o0 = __floats2bfloat162_rn(v[0], v[1]), o1 = __floats2bfloat162_rn(v[2], v[3]);
      out.x = *reinterpret_cast<uint32_t*>(&o0);
      out.y = *reinterpret_cast<uint32_t*>(&o1);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(M.y) + yo) = out;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) M.counters[pass * M.NB + nb] = 0;
}

// Debug: decode every tile to W[k][n] (FP16). One warp per tile.
template <int BITS>
__global__ void __launch_bounds__(256) decode_kernel(const __grid_constant__ DecodeArgs a) {
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const long long tile = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int TN = a.N / 16;
  if (tile >= (long long)(a.K / 16) * TN) return;
  const int tk = (int)(tile / TN), tn = (int)(tile % TN);
  LaneWindow<BITS> lw;
  lw.init(lane);
  uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
  lw.load(a.trellis + (long long)tk * a.stride + (long long)tn * (8 * BITS), raw);
  lw.align(raw, win);
  decode8<BITS>(win, af);
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int m = 0; m < 4; m++) {
    // register m holds slots i = 2m, 2m+1
    const int i = 2 * m;
    const int nl = g + 8 * ((i >> 1) & 1), kl = 2 * t + 8 * (i >> 2);
    const __half2 hv = *reinterpret_cast<const __half2*>(&af[m]);
    a.W[(long long)(16 * tk + kl) * a.N + 16 * tn + nl] = __low2half(hv);
    a.W[(long long)(16 * tk + kl + 1) * a.N + 16 * tn + nl] = __high2half(hv);
  }
}

// Kernel pointers for one bit width (defined in exl3_b<BITS>.cu).
struct KernelSet {
  const void* linear_rows[2];  // decode-rows family: NR = 1, 2 (8 warps)
  const void* linear_mid[4];   // mid-rows family: NR = 2, 4, 8, 16 (16 warps)
  const void* decode;
};

}  // namespace tfx
