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
// Summation order (a function of K alone, identical in every kernel, launch
//   shape, row count, group and column view): the K/16 tile rows are cut into
//   C chunks, C a power of two, chunk c = tiles [c*TK/C, (c+1)*TK/C) (floor).
//   A chunk's sum is one chain of m16n8k16 MMAs from zero in increasing k,
//   accumulated in FP32. The C chunk sums combine by a balanced binary tree in
//   chunk order: (c0+c1), (c2+c3), ... then pairs of those, up to the root.
//   Any power-of-two group of consecutive chunks is a subtree, so a warp, a CTA
//   or a set of CTAs (through the split-K scratch) can each own a subtree
//   without changing a bit. The pages fix the determinism (PR #1467, "The
//   arithmetic": the mid-M kernels keep the linear's K ranges, warp-order sums
//   and split-order partials), not the tree shape.
// Split-K combine, three forms with the same arithmetic:
//   * decode rows (default): the C CTAs of a 128-column block are one cluster;
//     each parks its chunk sums in shared memory and, after a cluster barrier,
//     folds some rows of the block from all C CTAs' shared memory;
//   * decode rows, `rows` variant: each CTA writes its subtree sum to a scratch
//     slab and one thread publishes it (fence + atomic increment of the
//     block's counter); the CTA that sees the last arrival folds the slabs,
//     rotates back, stores y and resets the counter to 0 (PR #1475, "What this
//     changes": the last arriving program resets counters[pass*NB + nb]);
//   * tensor core: units write slabs that a combine kernel folds.
//   No CTA ever spins on another CTA's progress (cluster barriers are
//   hardware barriers of co-scheduled CTAs).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tfx {

constexpr uint32_t kHashMul = 0x9E3779B1u;
constexpr uint32_t kHashAdd = 0x7F4A7C15u;
constexpr float kInvSqrt128 = 0.08838834764831845f;  // 1/sqrt(128) rounded to FP32
constexpr int kRowsPerPass = 128;
constexpr int kMaxChunks = 16;

struct Member {
  const uint32_t* trellis;  // first tile of this weight (or view)
  long long stride;         // uint32 words between tile rows
  const __half* svh;        // N
  const __half* suh;        // K (read by the decode-rows kernel when it rotates x itself)
  const uint2* xf;          // rotated x in B-fragment order (see xf_index)
  void* y;                  // output: element (r, n) at y + r*ldy + (n - col0), act dtype
  long long ldy;            // elements between output rows (N for a plain call)
  int col0;                 // first output column stored (0 for a plain call; a multiple of 8)
  float* partial;           // [pass][P][rp][N] FP32 subtree sums
  int* counters;            // [pass][NB]
  int N, NB;
  int C;                    // K chunks (power of two): defines the bits
  int G, log2G;             // chunks per unit: a warp (decode rows) or a CTA (mid rows)
  int P;                    // slabs per pass = C / G
  int TC;                   // 16-column tiles per CTA
  int arrivals;             // CTAs per (pass, 128-column block)
  int cta_begin;            // first blockIdx.x of this member
};

// How the decode-rows kernel folds a block's C chunk sums: in the block's
// cluster (distributed shared memory, two cluster barriers), through global
// slabs summed by the last CTA to arrive on the block's counter, or through
// global slabs summed by the combine kernel launched after it.
constexpr int kFoldCluster = 0, kFoldCounter = 1, kFoldCombine = 2;

struct LinearArgs {
  Member m[3];
  int count;
  int K, TK;    // K and K/16
  int rows;     // total rows
  int passes;   // ceil(rows / 128)
  int rp;       // row stride of a partial slab = min(rows, 128)
  int act;      // 0 FP16, 1 BF16
  long long items;  // work items of the warp-granular kernel (all members)
  int* err;         // device error word of the call
  long long spin;   // clock cycles a bounded wait polls before it gives up
  int box_rows;     // warp-granular kernel: tile rows per tensor copy of trellis words (H)
  int ring_boxes;   // warp-granular kernel: trellis copies in flight per warp (R, 1 or 2)
  int x_rows;       // warp-granular kernel: tile rows per x stage (the whole chunk, or H)
  int x_whole;      // warp-granular kernel: 1 if one x stage holds the whole chunk
  int fuse_rot;     // warp-granular kernel: 1 if each CTA rotates its chunk of x itself (few rows)
  int fold_mode;    // warp-granular kernel: how a block's chunk sums are folded (kFoldCluster,
                    // kFoldCounter, kFoldCombine)
  int early_arrive; // warp-granular kernel: 1 to arrive on the closing cluster barrier right after
                    // the fold's distributed loads (launches of many cluster waves)
  const void* x;    // the call's x (rows x K, act dtype), read when fuse_rot
  CUtensorMap tm[3];  // warp-granular kernel: member m's trellis as a 2-D tensor of uint32
                      // words (columns of the view x K/16 tile rows), box (NCOL*8*BITS, H)
};

struct RotArgs {
  const void* x;        // rows x K, act dtype
  const __half* suh[3]; // per member
  uint2* xf[3];         // per member output
  int count, rows, rows_pad, K, act;  // rows_pad = rows rounded up to 16 (padding rows are zero)
  int layout;           // 0: m16n8k16 B-fragment order (xf_index); 1: tensor-core core matrices (xc_byte)
  int rp_tc;            // rows per pass of layout 1
};

struct DecodeArgs {
  const uint32_t* trellis;
  long long stride;
  __half* W;  // K x N
  int K, N;
};

// The rotated x is stored in the order the m16n8k16 B operand is consumed:
// for 8-row group q, 16-row tile tk of K and lane l = 4g + t, one uint2 holds
// {x[8q+g][16tk+2t], x[8q+g][16tk+2t+1]} and {x[8q+g][16tk+2t+8], x[8q+g][16tk+2t+9]}.
// A warp reads the fragment of one (q, tk) as 256 contiguous bytes.
__host__ __device__ __forceinline__ long long xf_index(int q, int tk, int lane, int TK) {
  return ((long long)q * TK + tk) * 32 + lane;
}

// log2 of a power of two
__host__ __device__ __forceinline__ int ilog2_pow2(int C) {
#ifdef __CUDA_ARCH__
  return __ffs(C) - 1;
#else
  return __builtin_ctz((unsigned)C);
#endif
}
// First tile row of chunk c: floor(c * TK / C), C a power of two.
__host__ __device__ __forceinline__ int chunk_begin(int c, int TK, int C) {
  return (int)(((long long)c * TK) >> ilog2_pow2(C));
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// mbarrier and bulk-copy (TMA engine) primitives, CTA scope.
__device__ __forceinline__ uint32_t s_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(s_addr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(s_addr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(s_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (test_wait never suspends the thread, unlike try_wait).
__device__ __forceinline__ bool mbar_poll(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(s_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   s_addr(dst)),
               "l"(src), "r"(bytes), "r"(s_addr(b))
               : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Balanced binary tree over n values in index order: (v0+v1), (v2+v3), ...
template <int N>
__device__ __forceinline__ float tree_sum(float (&v)[N]) {
#pragma unroll
  for (int step = 1; step < N; step *= 2) {
#pragma unroll
    for (int i = 0; i + step < N; i += 2 * step) v[i] = v[i] + v[i + step];
  }
  return v[0];
}

// Tree over n (a power of two <= 16) floats at p[i*stride]; CG selects L2 loads.
template <bool CG>
__device__ __forceinline__ float tree_load(const float* p, long long stride, int n) {
  auto ld = [&](int i) { return CG ? __ldcg(p + i * stride) : p[i * stride]; };
  if (n == 1) return ld(0);
  if (n == 2) {
    float v[2] = {ld(0), ld(1)};
    return tree_sum<2>(v);
  }
  if (n == 4) {
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) v[i] = ld(i);
    return tree_sum<4>(v);
  }
  if (n == 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = ld(i);
    return tree_sum<8>(v);
  }
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = ld(i);
  return tree_sum<16>(v);
}

// Output columns n0 .. n0+3 (n0 a multiple of 4) of row r of member M, rounded
// to the output dtype. Element (r, n) sits at M.y + r*M.ldy + (n - M.col0);
// columns below M.col0 are not stored (col0 is a multiple of 8, so the four
// columns are kept or dropped together).
__device__ __forceinline__ void store_y4(const Member& M, int act, long long r, int n0, const float (&v)[4]) {
  if (n0 < M.col0) return;
  const long long yo = r * M.ldy + (n0 - M.col0);
  uint2 out;
  if (act == 0) {
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
// One output element (r, n) of member M (dropped below M.col0).
__device__ __forceinline__ void store_y1(const Member& M, int act, long long r, int n, float v) {
  if (n < M.col0) return;
  const long long yo = r * M.ldy + (n - M.col0);
  if (act == 0)
    reinterpret_cast<__half*>(M.y)[yo] = __float2half_rn(v);
  else
    reinterpret_cast<__nv_bfloat16*>(M.y)[yo] = __float2bfloat16_rn(v);
}

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

// ---------------------------------------------------------------------------
// Pieces of the input rotation and of the split-K combine shared by the
// standalone kernels and the fused decode-rows kernel (same arithmetic, same
// order, hence the same bits).

// x[r][128b + 4*lane .. +3] as FP32 (zeros for padding rows r >= rows).
__device__ __forceinline__ void rot_load(const RotArgs& a, int r, int b, int lane, float (&xv)[4]) {
  xv[0] = xv[1] = xv[2] = xv[3] = 0.f;
  if (r >= a.rows) return;
  const long long base = (long long)r * a.K + 128LL * b + 4 * lane;
  if (a.act == 0) {
    uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(a.x) + base);
    __half2 h0 = *reinterpret_cast<__half2*>(&u.x), h1 = *reinterpret_cast<__half2*>(&u.y);
    xv[0] = __low2float(h0); xv[1] = __high2float(h0); xv[2] = __low2float(h1); xv[3] = __high2float(h1);
  } else {
    uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + base);
    __nv_bfloat162 h0 = *reinterpret_cast<__nv_bfloat162*>(&u.x), h1 = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    xv[0] = __low2float(h0); xv[1] = __high2float(h0); xv[2] = __low2float(h1); xv[3] = __high2float(h1);
  }
}

// fp16(Hn(suh_m o x)) of one 128-block, the lane's 4 values as two half2.
// suh of member m for the lane's 4 elements of 128-block b.
__device__ __forceinline__ uint2 rot_suh(const RotArgs& a, int m, int b, int lane) {
  return *reinterpret_cast<const uint2*>(a.suh[m] + 128LL * b + 4 * lane);
}
__device__ __forceinline__ void rot_member_su(uint2 su, int lane, const float (&xv)[4], __half2 (&h)[2]) {
  __half2 s0 = *reinterpret_cast<__half2*>(&su.x), s1 = *reinterpret_cast<__half2*>(&su.y);
  float v[4] = {xv[0] * __low2float(s0), xv[1] * __high2float(s0), xv[2] * __low2float(s1), xv[3] * __high2float(s1)};
  fwht128(v, lane);
#pragma unroll
  for (int mm = 0; mm < 2; mm++)
    h[mm] = __halves2half2(__float2half_rn(v[2 * mm] * kInvSqrt128), __float2half_rn(v[2 * mm + 1] * kInvSqrt128));
}
__device__ __forceinline__ void rot_member(const RotArgs& a, int m, int b, int lane, const float (&xv)[4],
                                           __half2 (&h)[2]) {
  rot_member_su(rot_suh(a, m, b, lane), lane, xv, h);
}

// Store in B-fragment order: element k = 128b + 4*lane + e sits in tile 8b + lane/4
// at kk = 4*(lane%4) + e; the pair (kk, kk+1) for kk = 4*(lane%4) + 2m belongs to
// fragment lane 4g + 2*(lane%2) + m, register (lane%4) >= 2 (the k+8 half).
__device__ __forceinline__ void rot_store_frag(const RotArgs& a, int m, int r, int b, int lane, const __half2 (&h)[2]) {
  const int TK = a.K / 16;
  const int q = r >> 3, gq = r & 7;
  const int tk = 8 * b + (lane >> 2);
  const int reg = (lane & 3) >= 2 ? 1 : 0;
  uint32_t* out = reinterpret_cast<uint32_t*>(a.xf[m]);
#pragma unroll
  for (int mm = 0; mm < 2; mm++) {
    const int fl = 4 * gq + 2 * (lane & 1) + mm;
    out[xf_index(q, tk, fl, TK) * 2 + reg] = *reinterpret_cast<const uint32_t*>(&h[mm]);
  }
}

// Row r of the call, 128-column block nb of member M: fold the P slabs
// [pass][P][rp][N] as a balanced tree, rotate back (FWHT, 1/sqrt(128)), scale
// by svh, store y. One warp; the lane's 4 columns of every slab come in one
// 16-byte load, all P loads in flight at once.
template <int P>
__device__ __forceinline__ void combine_fold(const float* base, long long slab, float (&v)[4]) {
  float4 s[P];
#pragma unroll
  for (int p = 0; p < P; p++) s[p] = __ldcg(reinterpret_cast<const float4*>(base + p * slab));
  float t[4][P];
#pragma unroll
  for (int p = 0; p < P; p++) {
    t[0][p] = s[p].x;
    t[1][p] = s[p].y;
    t[2][p] = s[p].z;
    t[3][p] = s[p].w;
  }
#pragma unroll
  for (int e = 0; e < 4; e++) v[e] = tree_sum<P>(t[e]);
}

__device__ __forceinline__ void combine_item(const LinearArgs& a, const Member& M, int r, int nb, int RP, int lane) {
  const int pass = r / RP, rr = r - pass * RP;
  const int n0 = nb * 128 + 4 * lane;
  const long long slab = (long long)a.rp * M.N;
  const float* base = M.partial + (long long)pass * M.P * slab + (long long)rr * M.N + n0;
  float v[4];
  switch (M.P) {
    case 1: combine_fold<1>(base, slab, v); break;
    case 2: combine_fold<2>(base, slab, v); break;
    case 4: combine_fold<4>(base, slab, v); break;
    case 8: combine_fold<8>(base, slab, v); break;
    default: combine_fold<16>(base, slab, v); break;
  }
  fwht128(v, lane);
  float sv[4];
#pragma unroll
  for (int e = 0; e < 4; e++) sv[e] = __half2float(M.svh[n0 + e]);
#pragma unroll
  for (int e = 0; e < 4; e++) v[e] = (v[e] * kInvSqrt128) * sv[e];
  store_y4(M, a.act, r, n0, v);
}

// Words of one tile a lane needs: its 8 weights' windows span bits
// [8*lane*BITS, 8*lane*BITS + 7*BITS + 16), at most 2 words for BITS <= 4
// and 3 words above, counted from the word holding the first bit.
template <int BITS>
struct Geo {
  static constexpr int kWords = 8 * BITS;          // words per tile
  static constexpr int kRaw = BITS <= 4 ? 2 : 3;   // words a lane needs
  static constexpr int kSpan = 7 * BITS + 16;      // bits used after alignment
  static constexpr int kNorm = (kSpan + 31) / 32;  // words after alignment
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

// Where a lane's window starts in a tile and how to align it to bit 0.
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

// One thread publishes the CTA's slab (all threads wrote it before the barrier)
// and learns whether it was the last arrival of the block. Release: fence then
// relaxed atomic; acquire: fence after seeing the final count.
__device__ __forceinline__ bool arrive_last(int* counter, int arrivals, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(counter, 1);
    const bool last = old == arrivals - 1;
    if (last) __threadfence();
    *s_flag = last;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Last arrival of a 128-column block: fold the P slabs as a tree, rotate back
// (FWHT, 1/sqrt(128)), scale by svh and store y. One warp per row.
__device__ __forceinline__ void block_epilogue(const Member& M, const LinearArgs& a, int pass, int nb, int prow,
                                               int row0, int warp, int nwarps, int lane) {
  const int n0 = nb * 128 + 4 * lane;
  float sv[4];
#pragma unroll
  for (int e = 0; e < 4; e++) sv[e] = __half2float(M.svh[n0 + e]);
  const long long slab = (long long)a.rp * M.N;
  const float* base = M.partial + (long long)pass * M.P * slab + n0;
  for (int r = warp; r < prow; r += nwarps) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = tree_load<true>(base + (long long)r * M.N + e, slab, M.P);
    fwht128(v, lane);
#pragma unroll
    for (int e = 0; e < 4; e++) v[e] = (v[e] * kInvSqrt128) * sv[e];
    store_y4(M, a.act, row0 + r, n0, v);
  }
}

__device__ __forceinline__ const Member& pick_member_at(const LinearArgs& a, long long idx) {
  int mi = 0;
  if (a.count > 1 && idx >= a.m[1].cta_begin) mi = 1;
  if (a.count > 2 && idx >= a.m[2].cta_begin) mi = 2;
  return a.m[mi];
}
__device__ __forceinline__ const Member& pick_member(const LinearArgs& a) { return pick_member_at(a, blockIdx.x); }


// ---------------------------------------------------------------------------
// Decode-rows kernel (1..64 rows in row tiles of 8*NR, one pass). One CTA = WPC warps = WPC
// consecutive tile-columns of one 128-column block, all on the same chunk
// group; each warp owns G consecutive chunks of its tile-column (a subtree),
// runs their MMA chains one after the other and folds them in registers as the
// tree prescribes (a binary counter of subtree sums). The subtree sum goes to
// slab gidx. Small CTAs and a chunk grouping sized to the SM count keep the
// work of one launch spread evenly over the GPU. Each lane prefetches the
// trellis words and x fragments of the next PF tiles into registers; the word
// loads skip L1, which keeps x resident there.

// The words a lane needs from one tile. For BITS <= 4 a tile is at most 32
// words: each lane loads one word (word l) and takes the words it needs from
// their owners by shuffle. For BITS = 8 a lane loads words 2l, 2l+1 and takes
// 2l+2 from lane l+1. Other widths load their 3 words directly.
template <int BITS>
struct WordFetch {
  static constexpr int kOwn = BITS == 8 ? 2 : (BITS <= 4 ? 1 : Geo<BITS>::kRaw);
  __device__ __forceinline__ static void load(const uint32_t* __restrict__ tile, const LaneWindow<BITS>& lw, int lane,
                                              uint32_t (&own)[kOwn]) {
    if constexpr (BITS <= 4) {
      const int j = lane < 8 * BITS ? lane : 0;
      asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(own[0]) : "l"(tile + j));
    } else if constexpr (BITS == 8) {
      uint2 v;
      asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(tile + 2 * lane));
      own[0] = v.x;
      own[1] = v.y;
    } else {
      own[0] = __ldg(tile + lw.i0);
      own[1] = __ldg(tile + lw.i1);
      own[2] = __ldg(tile + lw.i2);
    }
  }
  __device__ __forceinline__ static void gather(const uint32_t (&own)[kOwn], const LaneWindow<BITS>& lw, int lane,
                                                uint32_t (&raw)[Geo<BITS>::kRaw]) {
    if constexpr (BITS == 4) {
      raw[0] = own[0];
      raw[1] = __shfl_sync(0xffffffffu, own[0], (lane + 1) & 31);
    } else if constexpr (BITS < 4) {
      raw[0] = __shfl_sync(0xffffffffu, own[0], lw.i0);
      raw[1] = __shfl_sync(0xffffffffu, own[0], lw.i1);
    } else if constexpr (BITS == 8) {
      raw[0] = own[0];
      raw[1] = own[1];
      raw[2] = __shfl_sync(0xffffffffu, own[0], (lane + 1) & 31);
    } else {
#pragma unroll
      for (int i = 0; i < Geo<BITS>::kRaw; i++) raw[i] = own[i];
    }
  }
};

// One decode-rows step: the lane's words of one tile -> A fragment -> NR MMAs.
template <int BITS, int NR>
__device__ __forceinline__ void rows_step(const uint32_t (&own)[WordFetch<BITS>::kOwn], const uint2 (&xc)[NR],
                                          const LaneWindow<BITS>& lw, int lane, float (&acc)[NR][4]) {
  uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
  WordFetch<BITS>::gather(own, lw, lane, raw);
  lw.align(raw, win);
  decode8<BITS>(win, af);
#pragma unroll
  for (int q = 0; q < NR; q++) mma16816(acc[q], af, xc[q].x, xc[q].y);
}

// The MMA chain of tiles [t0, t0+n) of one tile-column into acc (from zero).
template <int BITS, int NR, int PF>
__device__ __forceinline__ void rows_chain(const uint32_t* __restrict__ tp, long long wstride,
                                           const uint2* __restrict__ xp, long long xstride_q, int n,
                                           const LaneWindow<BITS>& lw, int lane, float (&acc)[NR][4]) {
  using WF = WordFetch<BITS>;
#pragma unroll
  for (int q = 0; q < NR; q++) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
  uint32_t own[PF][WF::kOwn];
  uint2 xr[PF][NR];
#pragma unroll
  for (int p = 0; p < PF; p++) {
    if (p < n) {
      WF::load(tp + p * wstride, lw, lane, own[p]);
#pragma unroll
      for (int q = 0; q < NR; q++) xr[p][q] = __ldcg(xp + q * xstride_q + 32 * p);
    }
  }
  int tk = 0;
  // full rounds: every tile of the round exists, its refill may not
  for (; tk + PF <= n; tk += PF) {
#pragma unroll
    for (int p = 0; p < PF; p++) {
      uint32_t oc[WF::kOwn];
      uint2 xc[NR];
#pragma unroll
      for (int i = 0; i < WF::kOwn; i++) oc[i] = own[p][i];
#pragma unroll
      for (int q = 0; q < NR; q++) xc[q] = xr[p][q];
      const int nx = tk + p + PF;
      if (nx < n) {
        WF::load(tp + nx * wstride, lw, lane, own[p]);
#pragma unroll
        for (int q = 0; q < NR; q++) xr[p][q] = __ldcg(xp + q * xstride_q + 32 * nx);
      }
      rows_step<BITS, NR>(oc, xc, lw, lane, acc);
    }
  }
  // tail: the last n % PF tiles are already in registers
#pragma unroll
  for (int p = 0; p < PF; p++)
    if (tk + p < n) rows_step<BITS, NR>(own[p], xr[p], lw, lane, acc);
}

constexpr int kRowsMaxLog2G = 3;  // up to 8 chunks per warp
constexpr int kRowsMaxRows = 64;  // the widest decode-rows row tile (NR = 8)
constexpr int kRowsTC = 2;        // tile-columns per decode-rows CTA
constexpr int kRowsGW = 4;        // warp groups per tile-column (consecutive chunk groups)

// CTA = kRowsTC x kRowsGW warps; warp (c, h) owns chunks [(gidx*GW + h)*G, +G)
// of tile-column c. Warp trees (registers + parked levels in shared memory),
// then a tree over the GW warps of a column in shared memory, give the CTA's
// subtree of GW*G chunks: slab gidx of P = C/(GW*G).
template <int BITS, int NR, int PF, int MINB>
__global__ void __launch_bounds__(kRowsTC * kRowsGW * 32, MINB)
    linear_rows_kernel(const __grid_constant__ LinearArgs a) {
  constexpr int WPC = kRowsTC * kRowsGW;
  // parked tree levels: up to 2^kRowsMaxLog2G chunks per warp at 1..16 rows;
  // wider row tiles run one chunk per warp (G = 1) and park nothing
  constexpr int kLev = NR <= 2 ? kRowsMaxLog2G : 0;
  __shared__ int s_last;
  __shared__ float lev[kLev ? WPC : 1][kLev ? kLev : 1][kLev ? NR * 4 : 1][32];
  __shared__ float red[kRowsTC][kRowsGW][NR * 8][16];
  griddep_wait();
  griddep_launch();
  const Member& M = pick_member(a);

  // one pass (rows <= 8*NR <= 64): blockIdx -> (column group of kRowsTC tile-columns, chunk group)
  const int local = blockIdx.x - M.cta_begin;
  const int gidx = local % M.P;
  const int colgrp = local / M.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int c = warp % kRowsTC, h = warp / kRowsTC;
  const int tn = colgrp * kRowsTC + c;
  const int nb = tn >> 3;
  const int prow = a.rows;
  const int GW = M.TC;  // warp groups in use (kRowsGW, or C when C < kRowsGW)

  if (h < GW) {
    LaneWindow<BITS> lw;
    lw.init(lane);
    const long long wstride = M.stride;
    const long long xstride_q = 32LL * a.TK;
    const uint32_t* col = M.trellis + (long long)tn * (8 * BITS);
    float acc[NR][4];
    for (int ci = 0; ci < M.G; ci++) {
      const int chunk = (gidx * GW + h) * M.G + ci;
      const int t0 = chunk_begin(chunk, a.TK, M.C), t1 = chunk_begin(chunk + 1, a.TK, M.C);
      rows_chain<BITS, NR, PF>(col + (long long)t0 * wstride, wstride, M.xf + xf_index(0, t0, lane, a.TK),
                               xstride_q, t1 - t0, lw, lane, acc);
      // while bit l of ci is set: acc = lev[l] + acc; then park acc at the first clear bit
      if constexpr (kLev > 0) {
        int l = 0;
        for (; l < kLev && ((ci >> l) & 1); l++) {
#pragma unroll
          for (int q = 0; q < NR; q++)
#pragma unroll
            for (int e = 0; e < 4; e++) acc[q][e] = lev[warp][l][q * 4 + e][lane] + acc[q][e];
        }
        if (ci + 1 < M.G) {
#pragma unroll
          for (int q = 0; q < NR; q++)
#pragma unroll
            for (int e = 0; e < 4; e++) lev[warp][l][q * 4 + e][lane] = acc[q][e];
        }
      }
    }
    // warp subtree -> red[c][h]: lane (g, t) holds (n = g | g+8, r = 8q + 2t | +1)
#pragma unroll
    for (int q = 0; q < NR; q++) {
      const int r0 = 8 * q + 2 * t;
      red[c][h][r0][g] = acc[q][0];
      red[c][h][r0 + 1][g] = acc[q][1];
      red[c][h][r0][g + 8] = acc[q][2];
      red[c][h][r0 + 1][g + 8] = acc[q][3];
    }
  }
  __syncthreads();

  // tree over the GW warp subtrees of each column -> slab gidx
  float* part = M.partial + (long long)gidx * a.rp * M.N + colgrp * (kRowsTC * 16);
  for (int idx = threadIdx.x; idx < prow * kRowsTC * 16; idx += WPC * 32) {
    const int r = idx / (kRowsTC * 16), cc = idx % (kRowsTC * 16);
    const int cw = cc >> 4, nl = cc & 15;
    part[(long long)r * M.N + cc] = tree_load<false>(&red[cw][0][r][nl], NR * 8 * 16, GW);
  }
  if (!arrive_last(&M.counters[nb], M.arrivals, &s_last)) return;
  block_epilogue(M, a, 0, nb, prow, 0, warp, WPC, lane);
  __syncthreads();
  if (threadIdx.x == 0) M.counters[nb] = 0;
}

// Warp-granular decode-rows kernel (1..64 rows, one pass). A CTA covers one
// 128-column block for one K chunk: 8/NCOL warps, warp w owning NCOL adjacent
// tile-columns, each running that chunk's MMA chain for them. The C CTAs of a
// block (its C chunks) form one thread-block cluster. Both operands are moved
// by the copy engine into shared memory:
//   * the warp's trellis words: before anything else, lane 0 asks for the
//     chain's tile rows as 2-D boxes of H rows x NCOL tiles (one tensor copy
//     per box) into the warp's own ring of R (1 or 2) boxes, so a whole SM's
//     share of a small layer is in flight from the first cycles; a finished
//     box is refilled with the box R further on;
//   * the rotated x of the chunk (written by the rotation kernel, so read only
//     after the wait on it): thread 0 bulk-copies the matching H tiles of x
//     fragments into the CTA's ring of R stages, shared by its warps; a stage
//     is refilled once every warp has arrived on its `empty` barrier.
// Split-K combine inside the cluster: every CTA parks its chain sums (rows x
// 128 FP32) in its own shared memory; after a cluster barrier, the CTA of
// chunk i folds rows i, i + C, ... : one warp per row reads the C chunk sums
// of the row from the C CTAs' shared memory (distributed shared memory),
// adds them as the chunk tree prescribes (a balanced binary tree in chunk
// order), rotates back (FWHT, 1/sqrt(128)), scales by svh and stores y. A
// second cluster barrier keeps every CTA's shared memory alive until all
// reads are done. No scratch, no counters, no second kernel.
constexpr long long kSpinClocks = 2000000000LL;  // default clock cycles before a wait gives up (about 1 s)

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// descheduled until it completes or about `ns` nanoseconds pass, so waiting
// warps leave the issue slots to the warps that decode.
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* b, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(s_addr(b)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase of the given parity, at most `spin` clock cycles (the
// launch's limit, kSpinClocks unless a test lowers it); false on a timeout.
// The wait spins on the non-blocking test: measured on GB300, a try_wait
// that finds the phase incomplete suspends the thread for a fixed slice
// (about half a microsecond) rather than until the phase completes, which
// made every producer/consumer hand-off cost that much.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity, long long spin) {
  if (mbar_poll(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_poll(b, parity))
    if (clock64() - t0 > spin) return false;
  return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          s_addr(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(s_addr(b))
      : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// 16 bytes at the same shared-memory offset in the CTA of cluster rank `rank`
__device__ __forceinline__ float4 ld_dsmem_f4(const void* local, int rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(s_addr(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// Fold the P chunk sums of one row (4 consecutive columns per lane) held by
// the cluster's CTAs at the same offset, as a balanced tree in chunk order.
template <int P>
__device__ __forceinline__ void cluster_fold(const float* local, float (&v)[4]) {
  float4 s[P];
#pragma unroll
  for (int p = 0; p < P; p++) s[p] = ld_dsmem_f4(local, p);
  float t[4][P];
#pragma unroll
  for (int p = 0; p < P; p++) {
    t[0][p] = s[p].x;
    t[1][p] = s[p].y;
    t[2][p] = s[p].z;
    t[3][p] = s[p].w;
  }
#pragma unroll
  for (int e = 0; e < 4; e++) v[e] = tree_sum<P>(t[e]);
}

// Rotate one row of a 128-column block back and store it: FWHT over the 128
// values (4 per lane), x 1/sqrt(128), x svh, round to the output dtype.
// sv4 holds the lane's 4 svh values (read before the caller's barriers, so
// that no global load sits on the epilogue's critical path).
__device__ __forceinline__ void rot_out_row(float (&v)[4], uint2 sv4, const Member& M, long long r, int n0, int act,
                                            int lane) {
  fwht128(v, lane);
  float sv[4];
  {
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sv4.x), s23 = *reinterpret_cast<const __half2*>(&sv4.y);
    sv[0] = __low2float(s01);
    sv[1] = __high2float(s01);
    sv[2] = __low2float(s23);
    sv[3] = __high2float(s23);
  }
#pragma unroll
  for (int e = 0; e < 4; e++) v[e] = (v[e] * kInvSqrt128) * sv[e];
  store_y4(M, act, r, n0, v);
}

// Shared memory of the warp-granular kernel: R stages of x (NR row groups x H
// tiles x 256 bytes) and, per warp, R boxes of H tile rows of NCOL tiles (each
// padded to 128 bytes); after the chains the same space holds the CTA's chain
// sums (rows x 128 FP32). Plus 128 bytes of alignment slack.
__host__ __device__ constexpr int warp_cta_warps(int ncol) { return 8 / ncol; }
__host__ __device__ constexpr int warp_row_bytes(int bits, int ncol) { return ncol * 32 * bits; }
__host__ __device__ inline int warp_box_bytes(int H, int bits, int ncol) {
  return (H * warp_row_bytes(bits, ncol) + 127) & ~127;
}
__host__ __device__ inline int warp_x_stage_bytes(int H, int nr) { return nr * H * 256; }
__host__ __device__ inline int warp_smem_bytes(int H, int R, int XH, int x_whole, int bits, int ncol, int nr,
                                               int rows) {
  const int ring = (x_whole ? 1 : R) * warp_x_stage_bytes(XH, nr) + R * warp_cta_warps(ncol) * warp_box_bytes(H, bits, ncol);
  const int park = rows * 128 * 4;
  return (ring > park ? ring : park) + 128;
}

template <int BITS, int NR, int NCOL>
__global__ void __launch_bounds__(32 * warp_cta_warps(NCOL)) linear_warp_kernel(const __grid_constant__ LinearArgs a) {
  constexpr int W = warp_cta_warps(NCOL);
  constexpr int RB = warp_row_bytes(BITS, NCOL);
  constexpr int RW = RB / 4;
  extern __shared__ unsigned char wsm[];
  __shared__ __align__(8) uint64_t wfull[W][2];
  __shared__ __align__(8) uint64_t xfull[2], xempty[2];
  __shared__ int s_dead, s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long cta = blockIdx.x;
  int mi = 0;
  if (a.count > 1 && cta >= a.m[1].cta_begin) mi = 1;
  if (a.count > 2 && cta >= a.m[2].cta_begin) mi = 2;
  const Member& M = a.m[mi];
  const int local = (int)(cta - M.cta_begin);
  const int lc = ilog2_pow2(M.C);
  const int chunk = local & (M.C - 1);  // = this CTA's rank in its cluster
  const int nb = local >> lc;           // 128-column block
  const int tn0 = nb * 8 + warp * NCOL;
  const int t0 = chunk_begin(chunk, a.TK, M.C), n = chunk_begin(chunk + 1, a.TK, M.C) - t0;
  const int H = a.box_rows, R = a.ring_boxes, XH = a.x_rows;
  const bool xw = a.x_whole != 0;
  const int nbox = (n + H - 1) / H;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(wsm) + 127) & ~uintptr_t(127));
  const int XS = warp_x_stage_bytes(XH, NR);
  const int BB = warp_box_bytes(H, BITS, NCOL);
  const uint2* xs = reinterpret_cast<const uint2*>(base);
  uint32_t* ring = reinterpret_cast<uint32_t*>(base + (xw ? 1 : R) * XS + warp * R * BB);
  // the trellis words are the caller's and no kernel of the layer writes them:
  // ask for them before waiting on the rotation kernel
  if (lane == 0) {
    mbar_init(&wfull[warp][0], 1);
    mbar_init(&wfull[warp][1], 1);
    if (warp == 0) {
      mbar_init(&xfull[0], 1);
      mbar_init(&xfull[1], 1);
      mbar_init(&xempty[0], W);
      mbar_init(&xempty[1], W);
      s_dead = 0;
    }
    fence_mbar_init();
    for (int b = 0; b < R && b < nbox; b++) {
      mbar_expect_tx(&wfull[warp][b], (uint32_t)(H * RB));
      tma_load_2d(ring + b * (BB / 4), &a.tm[mi], tn0 * 8 * BITS, t0 + b * H, &wfull[warp][b]);
    }
  }
  __syncthreads();
  // the dependent launch is triggered after the chain loop, not here: an
  // early trigger lets the next kernel's CTAs occupy SM resources for the
  // whole kernel
  griddep_wait();
  // x stage of box b: the chunk's tiles [b*H, min(n, (b+1)*H)) of every row
  // group q (or, with a whole-chunk stage, all n tiles at once), each one
  // contiguous run of 256 bytes per tile in the fragment layout
  auto load_x = [&](int b) {
    const int rows_b = xw ? n : min(H, n - b * H);
    const int st = xw ? 0 : (b & (R - 1));
    mbar_expect_tx(&xfull[st], (uint32_t)(NR * rows_b * 256));
    for (int q = 0; q < NR; q++)
      bulk_g2s(base + st * XS + q * XH * 256, M.xf + xf_index(q, t0 + (xw ? 0 : b * H), 0, a.TK),
               (uint32_t)(rows_b * 256), &xfull[st]);
  };
  const bool fuse = a.fuse_rot != 0;  // only with a whole-chunk x stage (host-checked)
  if (fuse) {
    // rotate the chunk's x here instead of copying what the rotation kernel
    // wrote: the 128-blocks overlapping the chunk, the call's real rows, the
    // same arithmetic as the rotation kernel (rot_load, rot_member) and the
    // same fragment order, into the zeroed x stage
    RotArgs ra = {};
    ra.x = a.x;
    ra.suh[0] = M.suh;
    ra.rows = a.rows;
    ra.K = a.K;
    ra.act = a.act;
    uint4* z = reinterpret_cast<uint4*>(base);
    for (int i = threadIdx.x; i < XS / 16; i += blockDim.x) z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const int b0 = (t0 * 16) >> 7, b1 = ((t0 + n) * 16 - 1) >> 7;
    const int items = (b1 - b0 + 1) * a.rows;
    uint32_t* xs32 = reinterpret_cast<uint32_t*>(base);
    for (int it = warp; it < items; it += W) {
      const int r = it / (b1 - b0 + 1), b = b0 + it % (b1 - b0 + 1);
      float xv[4];
      __half2 h[2];
      rot_load(ra, r, b, lane, xv);
      rot_member(ra, 0, b, lane, xv, h);
      const int q = r >> 3, gq = r & 7;
      const int tk = 8 * b + (lane >> 2);
      const int reg = (lane & 3) >= 2 ? 1 : 0;
      if (tk >= t0 && tk < t0 + n)
#pragma unroll
        for (int mm = 0; mm < 2; mm++) {
          const int fl = 4 * gq + 2 * (lane & 1) + mm;
          xs32[((q * XH + (tk - t0)) * 32 + fl) * 2 + reg] = *reinterpret_cast<const uint32_t*>(&h[mm]);
        }
    }
    __syncthreads();
  } else if (threadIdx.x == 0) {
    for (int b = 0; b < (xw ? 1 : R) && b < nbox; b++) load_x(b);
  }
  float acc[NCOL][NR][4];
#pragma unroll
  for (int c = 0; c < NCOL; c++)
#pragma unroll
    for (int q = 0; q < NR; q++) acc[c][q][0] = acc[c][q][1] = acc[c][q][2] = acc[c][q][3] = 0.f;
  LaneWindow<BITS> lw;
  lw.init(lane);
  // svh of this lane's 4 output columns for the warps that fold a row at the
  // end (svh is 16-byte aligned and a view starts on a 128-column block). With
  // one row group (rows <= 8) it is read now, so that no global load sits on
  // the epilogue's critical path: at one row the CTA of chunk 0 folds the
  // whole row after the others wait for it (measured 0.5 us per call)
  uint2 sv4 = make_uint2(0u, 0u);
  if constexpr (NR == 1)
    if (chunk + warp * M.C < a.rows) sv4 = *reinterpret_cast<const uint2*>(M.svh + nb * 128 + 4 * lane);
  bool alive = true;
  for (int b = 0; b < nbox && alive; b++) {
    const int st = b & (R - 1);
    const uint32_t par = (uint32_t)(b / R) & 1u;
    bool ok = mbar_wait_bounded(&wfull[warp][st], par, a.spin);
    if (!fuse && (xw ? b == 0 : true)) ok = ok && mbar_wait_bounded(&xfull[xw ? 0 : st], xw ? 0u : par, a.spin);
    if (!__all_sync(0xffffffffu, ok)) {
      alive = false;
      break;
    }
    const uint32_t* wr = ring + st * (BB / 4);
    const uint2* xr = xw ? xs + lane + b * H * 32 : xs + st * (XS / 8) + lane;
    const int rows_b = min(H, n - b * H);
    // four tile rows per unrolled body (measured on GB300 at 64 registers, no
    // spills: against two, 5120 x 5120 at 16 rows 16.2 -> 15.9 us, the LM head
    // at 1 row 442 -> 424 us; five and eight were slower)
#pragma unroll 4
    for (int r = 0; r < rows_b; r++) {
      const uint32_t* rr = wr + r * RW;
      uint32_t raw[NCOL][Geo<BITS>::kRaw];
#pragma unroll
      for (int c = 0; c < NCOL; c++) {
        raw[c][0] = rr[c * 8 * BITS + lw.i0];
        raw[c][1] = rr[c * 8 * BITS + lw.i1];
        if constexpr (Geo<BITS>::kRaw > 2) raw[c][2] = rr[c * 8 * BITS + lw.i2];
      }
      uint2 xc[NR];
#pragma unroll
      for (int q = 0; q < NR; q++) xc[q] = xr[(q * XH + r) * 32];
#pragma unroll
      for (int c = 0; c < NCOL; c++) {
        uint32_t win[Geo<BITS>::kNorm + 1], af[4];
        lw.align(raw[c], win);
        decode8<BITS>(win, af);
#pragma unroll
        for (int q = 0; q < NR; q++) mma16816(acc[c][q], af, xc[q].x, xc[q].y);
      }
    }
    if (b + R < nbox) {
      // hand the box back: this warp's words to its own next copy, the x
      // stage to thread 0 once every warp has arrived
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_expect_tx(&wfull[warp][st], (uint32_t)(H * RB));
        tma_load_2d(ring + st * (BB / 4), &a.tm[mi], tn0 * 8 * BITS, t0 + (b + R) * H, &wfull[warp][st]);
        if (!xw) {
          mbar_arrive(&xempty[st]);
          if (warp == 0) {
            if (mbar_wait_bounded(&xempty[st], par, a.spin))
              load_x(b + R);
            else
              s_dead = 1;
          }
        }
      }
    }
  }
  if (!alive && lane == 0) s_dead = 1;
  // with programmatic dependent launch, the next kernel may start launching
  // once every CTA is past its chain loop: all of this kernel's CTAs are then
  // resident, so the dependents' CTAs (which wait for this grid before they
  // read its output) only overlap the cluster epilogue
  griddep_launch();
  __syncthreads();
  const bool dead = s_dead != 0;
  if (dead) {
    // a copy never completed: report it and give copies still in flight time
    // to land in this CTA's shared memory; the cluster still meets at both
    // barriers, and nothing is written
    if (threadIdx.x == 0) atomicExch(a.err, 3);
    const long long w0 = clock64();
    while (clock64() - w0 < 2000000) {
    }
  }
  if (a.fold_mode != kFoldCluster) {
    // the launch has no clusters: this chunk's sums go to the block's slab
    // [chunk][row][N]; with kFoldCounter the block's last CTA to arrive on its
    // counter folds the C slabs in chunk order (the same balanced tree),
    // rotates back, stores y and resets the counter (PR #1475's split-K form),
    // with kFoldCombine the combine kernel does that for every (row, block) in
    // parallel; either way no CTA waits for another
    if (!dead) {
      float* slab = M.partial + (long long)chunk * a.rp * M.N + nb * 128;
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int c = 0; c < NCOL; c++)
#pragma unroll
        for (int q = 0; q < NR; q++) {
          const int r0 = 8 * q + 2 * t;
          float* pc = slab + (warp * NCOL + c) * 16 + g;
          if (r0 < a.rows) {
            __stcg(pc + (long long)r0 * M.N, acc[c][q][0]);
            __stcg(pc + (long long)r0 * M.N + 8, acc[c][q][2]);
          }
          if (r0 + 1 < a.rows) {
            __stcg(pc + (long long)(r0 + 1) * M.N, acc[c][q][1]);
            __stcg(pc + (long long)(r0 + 1) * M.N + 8, acc[c][q][3]);
          }
        }
    }
    if (a.fold_mode == kFoldCounter && arrive_last(M.counters + nb, M.C, &s_last)) {
      block_epilogue(M, a, 0, nb, a.rows, 0, warp, W, lane);
      if (threadIdx.x == 0) M.counters[nb] = 0;
    }
    return;
  }
  // park the chain sums: park[r][128] FP32, lane (g, t) holds (row 8q + 2t | +1,
  // column g | g + 8) of tile-column warp*NCOL + c
  float* park = reinterpret_cast<float*>(base);
  {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int c = 0; c < NCOL; c++)
#pragma unroll
      for (int q = 0; q < NR; q++) {
        const int r0 = 8 * q + 2 * t;
        float* pc = park + (warp * NCOL + c) * 16 + g;
        if (r0 < a.rows) {
          pc[r0 * 128] = acc[c][q][0];
          pc[r0 * 128 + 8] = acc[c][q][2];
        }
        if (r0 + 1 < a.rows) {
          pc[(r0 + 1) * 128] = acc[c][q][1];
          pc[(r0 + 1) * 128 + 8] = acc[c][q][3];
        }
      }
  }
  cluster_sync();
  // with more than one row group, svh is read here, where its latency overlaps
  // the distributed shared-memory loads of the fold
  if constexpr (NR > 1)
    if (chunk + warp * M.C < a.rows) sv4 = *reinterpret_cast<const uint2*>(M.svh + nb * 128 + 4 * lane);
  // rows chunk, chunk + C, ... of this block: one warp per row. No CTA of the
  // cluster may exit while another still reads its shared memory: the closing
  // cluster barrier. With early_arrive a warp arrives on it as soon as its
  // last distributed load has returned and waits only at the end, so the
  // CTAs that fold no row leave (and free their SM slots for the next cluster
  // wave) while the folding warps rotate and store; measured on GB300 this
  // helps launches of many waves (LM head at 1 row 455 -> 442 us) and costs
  // single-wave ones about 0.25 us, so the host sets it per launch
  bool arrived = a.early_arrive == 0;
  for (int r = chunk + warp * M.C; r < a.rows && !dead; r += W * M.C) {
    float v[4];
    const float* src = park + r * 128 + 4 * lane;
    switch (M.C) {
      case 1: cluster_fold<1>(src, v); break;
      case 2: cluster_fold<2>(src, v); break;
      case 4: cluster_fold<4>(src, v); break;
      case 8: cluster_fold<8>(src, v); break;
      default: cluster_fold<16>(src, v); break;
    }
    if (!arrived && r + W * M.C >= a.rows) {
      cluster_arrive();
      arrived = true;
    }
    rot_out_row(v, sv4, M, r, nb * 128 + 4 * lane, a.act, lane);
  }
  if (!arrived || a.early_arrive == 0) cluster_arrive();
  cluster_wait();
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

// Decode-rate probe: the decode rule's arithmetic at full occupancy with no
// global-memory traffic. Each warp decodes `tiles` tiles whose words it reads
// from a table of 64 tiles in shared memory (as the decode-rows kernels read
// their staged words) and feeds each decoded A fragment to one m16n8k16 MMA;
// one float per warp goes to `sink` so that nothing is optimised away. Timed
// by the caller, it gives the decoded weights per second this GPU sustains
// for the rule: the ALU roofline of the decode-bound calls.
constexpr int kRateWarps = 8;
constexpr int kRateCtasPerSm = 8;
struct RateArgs {
  int tiles;
  float* sink;  // gridDim.x * kRateWarps floats
};

template <int BITS>
__global__ void __launch_bounds__(kRateWarps * 32) decode_rate_kernel(const __grid_constant__ RateArgs a) {
  __shared__ uint32_t table[64 * 8 * BITS];
  for (int i = threadIdx.x; i < 64 * 8 * BITS; i += blockDim.x)
    table[i] = ((uint32_t)i * 2654435761u) ^ ((uint32_t)blockIdx.x * 40503u);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  LaneWindow<BITS> lw;
  lw.init(lane);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t xb = 0x3c003c00u;  // FP16 ones
  for (int t = 0; t < a.tiles; t++) {
    const uint32_t* tile = table + ((t + warp) & 63) * (8 * BITS);
    uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
    raw[0] = tile[lw.i0];
    raw[1] = tile[lw.i1];
    if constexpr (Geo<BITS>::kRaw > 2) raw[2] = tile[lw.i2];
    lw.align(raw, win);
    decode8<BITS>(win, af);
    mma16816(acc, af, xb, xb);
  }
  if (lane == 0) a.sink[blockIdx.x * kRateWarps + warp] = acc[0] + acc[1] + acc[2] + acc[3];
}

// Kernel pointers for one bit width (defined in exl3_bits.cu).
struct KernelSet {
  const void* linear_rows[4];  // decode-rows family: NR = 1, 2, 4, 8 (8, 16, 32, 64 rows)
  const void* linear_warp[4];  // warp-granular decode-rows kernel, same row tiles
  const void* linear_tc;       // tensor-core family: any row count, persistent
  const void* decode;
  const void* decode_rate;     // decode-rate probe
};

}  // namespace tfx
