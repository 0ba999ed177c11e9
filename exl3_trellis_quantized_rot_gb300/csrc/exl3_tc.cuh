// Tensor-core (tcgen05) mid-rows kernel of the EXL3 trellis linear for sm_103a.
//
// D[n][r] = sum_k W[k][n] * xr[r][k] per 128-column block with
//   A = decoded weights, M = 128 output columns, K-major, in shared memory;
//   B = rotated x rows of one 64-row pass, K-major, bulk-copied to shared memory;
//   D = FP32 accumulator in tensor memory (TMEM lane = output column, column = row).
// tcgen05.mma kind::f16 with FP32 accumulation returns the same bits as the
// m16n8k16 mma.sync chain of the decode-rows kernel for the same 16-wide k
// steps (measured on GB300 at N = 16..256), so both families keep the chunk
// tree's bits (see exl3_kernels.cuh).
//
// Shared-memory operand layout (no swizzle): 8x8 FP16 core matrices of 128 B,
// row-major inside; core (row group gr, k half kh) at (2*gr + kh) * 128 bytes,
// i.e. 128 B between k halves and 256 B between row groups.
//
// Roles in one CTA (17 warps): 16 decode warps in two groups (even / odd
// k-steps, one tile per warp per step, each group owning one A buffer) and a
// control warp whose lane 0 issues the bulk copies and, strictly in step
// order, the MMAs. Chunk c accumulates into TMEM region cur[c&1]; once its
// last MMA completes the decode warps fold it into the chunk tree (levels
// parked in TMEM) while chunk c+1 accumulates. Every wait is bounded: on a
// timeout the kernel records an error, stops issuing work and exits after
// releasing TMEM.
#pragma once
#include "exl3_kernels.cuh"

namespace tfx {

constexpr int kTcRowsPerPass = 64;  // rows per pass (N of the MMA, rounded up to 16)
constexpr int kTcDecodeWarps = 16;
constexpr int kTcThreads = (kTcDecodeWarps + 1) * 32;
constexpr int kTcSW = 24;                 // bulk-copy ring stages (one k-step each)
constexpr int kTcXStage = kTcRowsPerPass * 32;  // x bytes per k-step: N rows x 16 k x 2 B
constexpr int kTcAStage = 128 * 32;        // A bytes per k-step
constexpr int kTcAB = 4;                   // A buffers (decode group g uses g, g+2)
constexpr int kTcLag = 8;                  // a stage is refilled 8 steps after its MMA was issued
constexpr int kTcMaxLevels = 4;            // chunk tree levels parked in TMEM (C <= 16)
constexpr long long kTcSpin = 2000000000LL;  // clock cycles before a wait gives up
constexpr size_t kTcDynSmem = 120 * 1024;     // >= the rings; also keeps one CTA (one TMEM allocation) per SM

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
// try_wait may suspend the thread (here up to 0.1 ms) until the phase completes.
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(s_addr(b)), "r"(parity), "r"(100000)
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity to complete, at most kTcSpin cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err) {
  const long long t0 = clock64();
  while (!mbar_test(b, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kTcSpin) {
      *abort_flag = 1;
      atomicExch(err, 1);
      return false;
    }
  }
  return true;
}
// The same wait taken by all 32 lanes of a warp, with one warp-uniform outcome.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err) {
  const bool ok = mbar_wait(b, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok) != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   s_addr(dst)),
               "l"(src), "r"(bytes), "r"(s_addr(b))
               : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major, no swizzle: leading (k) byte offset 128, stride (row group) byte offset 256.
__device__ __forceinline__ uint64_t umma_desc(const void* p) {
  uint64_t d = (uint64_t)((s_addr(p) & 0x3FFFF) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(256 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// kind::f16: D FP32, A and B FP16, both K-major, M = 128.
__host__ __device__ constexpr uint32_t umma_idesc(int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_addr(b))
               : "memory");
}
// 4 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
               "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Rotated x in the tensor-core layout: element (r, k) at byte
// ((tk*Q + r/8)*2 + (k%16)/8)*128 + (r%8)*16 + (k%8)*2, Q = padded rows / 8,
// so the 64 rows of one pass at one k-step are 2 KB contiguous.
__host__ __device__ __forceinline__ long long xc_byte(int r, int k, int Q) {
  const int tk = k >> 4, kk = k & 15;
  return (((long long)tk * Q + (r >> 3)) * 2 + (kk >> 3)) * 128 + (r & 7) * 16 + (kk & 7) * 2;
}

struct TcArgs {
  LinearArgs la;
  int Q;     // padded rows / 8
  int* err;  // device error word: set to 1 when a wait timed out
};

template <int BITS>
__global__ void __launch_bounds__(kTcThreads, 1) linear_tc_kernel(const __grid_constant__ TcArgs ta) {
  const LinearArgs& a = ta.la;
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sX = dsm;                                 // [kTcSW][kTcXStage]
  unsigned char* sA = dsm + kTcSW * kTcXStage;             // [kTcAB][kTcAStage]
  unsigned char* sW = sA + kTcAB * kTcAStage;              // [kTcSW][8 tiles][8*BITS words]
  __shared__ __align__(8) uint64_t full[kTcSW], slot_free[kTcSW], a_ready[kTcAB], a_free[kTcAB], chunk_done[2],
      fold_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;

  griddep_wait();
  griddep_launch();
  const Member& M = pick_member(a);
  int local = blockIdx.x - M.cta_begin;
  const int pass = local % a.passes;
  local /= a.passes;
  const int gidx = local % M.P;
  const int nb = local / M.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = pass * kTcRowsPerPass;
  const int prow = min(kTcRowsPerPass, a.rows - row0);
  const int NM = (prow + 15) & ~15;  // MMA N
  const int G = M.G;
  const int c0 = gidx * G;  // first chunk of this CTA
  // total steps of the CTA's chunks
  const int tbeg = chunk_begin(c0, a.TK, M.C), tend = chunk_begin(c0 + G, a.TK, M.C);
  const int nsteps = tend - tbeg;
  // TMEM: two accumulator regions plus log2(G) parked tree levels, NM columns each
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)((2 + M.log2G) * NM)) tmem_cols *= 2;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kTcSW; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&slot_free[i], 1);
    }
    for (int i = 0; i < kTcAB; i++) {
      mbar_init(&a_ready[i], 8);
      mbar_init(&a_free[i], 1);
    }
    for (int i = 0; i < 2; i++) {
      mbar_init(&chunk_done[i], 1);
      mbar_init(&fold_done[i], kTcDecodeWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(&s_tmem)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t wbytes = 8 * 32 * BITS;        // one tile row of the block
  const uint32_t xbytes = (uint32_t)NM * 32;     // the pass's rows at one k-step
  const uint32_t idesc = umma_idesc(NM);
  const unsigned char* xsrc = reinterpret_cast<const unsigned char*>(M.xf) + ((long long)(row0 >> 3) * 2) * 128;
  const uint32_t* wsrc = M.trellis + (long long)nb * (64 * BITS);

  if (warp == kTcDecodeWarps) {
    // ---------------- control warp: bulk copies and MMAs in step order
    if (lane == 0) {
      auto issue = [&](int i) {
        const int s = i % kTcSW, tk = tbeg + i;
        mbar_expect_tx(&full[s], wbytes + xbytes);
        bulk_g2s(sW + s * (8 * 32 * BITS), wsrc + (long long)tk * M.stride, wbytes, &full[s]);
        bulk_g2s(sX + s * kTcXStage, xsrc + (long long)tk * ta.Q * 256, xbytes, &full[s]);
      };
      for (int i = 0; i < kTcSW && i < nsteps; i++) issue(i);
      int ci = 0;                                    // current chunk (relative)
      int cnext = chunk_begin(c0 + 1, a.TK, M.C) - tbeg;  // first step of the next chunk
      int cfirst = 0;
      for (int i = 0; i < nsteps && !s_abort; i++) {
        if (i == cnext) {
          ci++;
          cfirst = i;
          cnext = chunk_begin(c0 + ci + 1, a.TK, M.C) - tbeg;
          // chunk ci reuses region cur[ci&1]: its previous user (chunk ci-2) must be folded
          if (ci >= 2 && !mbar_wait(&fold_done[ci & 1], ((ci - 2) >> 1) & 1, &s_abort, ta.err)) break;
        }
        const int ab = i % kTcAB, s = i % kTcSW;
        if (!mbar_wait(&a_ready[ab], (i / kTcAB) & 1, &s_abort, ta.err)) break;
        tc_fence_after();
        umma_f16(tmem + (uint32_t)((ci & 1) * NM), umma_desc(sA + ab * kTcAStage), umma_desc(sX + s * kTcXStage),
                 idesc, i != cfirst ? 1u : 0u);
        umma_commit(&a_free[ab]);
        umma_commit(&slot_free[s]);
        if (i + 1 == cnext) umma_commit(&chunk_done[ci & 1]);
        // refill the stage of step i-kTcLag once its MMA has completed
        if (i >= kTcLag && i - kTcLag + kTcSW < nsteps) {
          const int sp = (i - kTcLag) % kTcSW;
          if (!mbar_wait(&slot_free[sp], ((i - kTcLag) / kTcSW) & 1, &s_abort, ta.err)) break;
          issue(i - kTcLag + kTcSW);
        }
      }
      if (s_abort) {
        // let copies already in flight land before the CTA's shared memory goes away
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
      }
    }
  } else {
    // ---------------- decode warps
    const int dg = warp >> 3, j = warp & 7;  // group, tile-column within the block
    LaneWindow<BITS> lw;
    lw.init(lane);
    const int g = lane >> 2, t = lane & 3;
    // A-fragment register m of tile j -> byte offset of its 4-byte pair in the core-matrix layout
    const int off0 = 512 * j + 16 * g + 4 * t;
    const int lg = warp & 3, cq = warp >> 2;  // TMEM lane group, column quarter (for the fold)
    const int qcols = NM >> 2;                // columns per warp in the fold
    float res[16];                            // this warp's share of the CTA's subtree after the last fold
    int chunk_of_next_fold = 0;
    int cnext_dec = chunk_begin(c0 + 1, a.TK, M.C) - tbeg;
    int cdec = 0;  // chunk of the step being decoded

    // fold of chunk cf (relative): merge cur[cf&1] into the tree levels
    auto fold = [&](int cf) {
      if (!mbar_wait_warp(&chunk_done[cf & 1], (cf >> 1) & 1, &s_abort, ta.err)) return;
      tc_fence_after();
      const uint32_t lane_base = (uint32_t)(lg * 32) << 16;
      for (int cc = 0; cc < qcols; cc += 4) {
        const uint32_t col = (uint32_t)(cq * qcols + cc);
        float v[4];
        tmem_ld4(tmem + lane_base + (uint32_t)((cf & 1) * NM) + col, v);
        int l = 0;
        for (; l < kTcMaxLevels && ((cf >> l) & 1); l++) {
          float u[4];
          tmem_ld4(tmem + lane_base + (uint32_t)((2 + l) * NM) + col, u);
#pragma unroll
          for (int e = 0; e < 4; e++) v[e] = u[e] + v[e];
        }
        if (cf + 1 < G) {
          tmem_st4(tmem + lane_base + (uint32_t)((2 + l) * NM) + col, v);
        } else {
#pragma unroll
          for (int e = 0; e < 4; e++) res[cc + e] = v[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&fold_done[cf & 1]);
    };

    for (int i = dg; i < nsteps; i += 2) {
      if (__any_sync(0xffffffffu, s_abort)) break;
      while (i >= cnext_dec) {
        cdec++;
        cnext_dec = chunk_begin(c0 + cdec + 1, a.TK, M.C) - tbeg;
      }
      // fold finished chunks once this warp has moved past them (chunk c is done
      // when this warp decodes a step of chunk c+1)
      while (chunk_of_next_fold < cdec) fold(chunk_of_next_fold++);
      const int s = i % kTcSW, ab = i % kTcAB;
      if (!mbar_wait_warp(&full[s], (i / kTcSW) & 1, &s_abort, ta.err)) break;
      if (i >= kTcAB && !mbar_wait_warp(&a_free[ab], ((i - kTcAB) / kTcAB) & 1, &s_abort, ta.err)) break;
      const uint32_t* tw = reinterpret_cast<const uint32_t*>(sW + s * (8 * 32 * BITS)) + j * (8 * BITS);
      uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
      raw[0] = tw[lw.i0];
      raw[1] = tw[lw.i1];
      if constexpr (Geo<BITS>::kRaw > 2) raw[2] = tw[lw.i2];
      lw.align(raw, win);
      decode8<BITS>(win, af);
      unsigned char* abuf = sA + ab * kTcAStage;
      *reinterpret_cast<uint32_t*>(abuf + off0) = af[0];        // n = g,   k = 2t..
      *reinterpret_cast<uint32_t*>(abuf + off0 + 256) = af[1];  // n = g+8, k = 2t..
      *reinterpret_cast<uint32_t*>(abuf + off0 + 128) = af[2];  // n = g,   k = 2t+8..
      *reinterpret_cast<uint32_t*>(abuf + off0 + 384) = af[3];  // n = g+8, k = 2t+8..
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_ready[ab]);
    }
    while (!__any_sync(0xffffffffu, s_abort) && chunk_of_next_fold < G) fold(chunk_of_next_fold++);

    // subtree sum -> slab gidx: TMEM lane = column 32*lg + lane, columns = rows
    if (!__any_sync(0xffffffffu, s_abort)) {
      float* part = M.partial + ((long long)pass * M.P + gidx) * a.rp * M.N + nb * 128 + lg * 32 + lane;
      for (int cc = 0; cc < qcols; cc++) {
        const int r = cq * qcols + cc;
        if (r < prow) part[(long long)r * M.N] = res[cc];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
  if (s_abort) return;
  if (!arrive_last(&M.counters[pass * M.NB + nb], M.arrivals, &s_last)) return;
  block_epilogue(M, a, pass, nb, prow, row0, warp, kTcDecodeWarps + 1, lane);
  __syncthreads();
  if (threadIdx.x == 0) M.counters[pass * M.NB + nb] = 0;
}

}  // namespace tfx
