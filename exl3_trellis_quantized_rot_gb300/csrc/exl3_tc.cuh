// Tensor-core (tcgen05) mid-rows kernel of the EXL3 trellis linear for sm_103a.
//
// D[n][r] = sum_k W[k][n] * xr[r][k] per 128-column block with
//   A = decoded weights, M = 128 output columns, K-major, in shared memory;
//   B = rotated x rows of one pass (up to 128 rows), K-major, bulk-copied to shared memory;
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
// The kernel is persistent: one CTA per SM walks the work units
// (member, pass, 128-column block, chunk group) in a fixed stride. The work
// of a unit is cut into stages of kTcSK k-steps that flow through warp roles:
//   warps 0..15   decode: load their tiles' words straight from global memory
//                 into a ring of register slots (up to two stages ahead) and
//                 turn 4 tiles per stage into FP16 A operands;
//   warps 16..19  fold: merge each finished chunk into the chunk tree (levels
//                 parked in TMEM), then write the unit's output: the whole
//                 rot_out epilogue when one unit covers all C chunks, else its
//                 FP32 slab, which tc_combine_kernel folds afterwards;
//   warp 20       issues the MMAs strictly in k order (lane 0);
//   warp 21       bulk-copies the x rows of each stage (lanes 0..3, a slice each).
// The decode warps hand a filled A buffer to the MMA warp, and the fold warps
// hand a folded TMEM region back to it, through hardware named barriers
// (waiting warps are descheduled, nothing polls). Completions of the
// asynchronous units (bulk copies, MMAs) are mbarriers that lane 0 of each
// waiting warp polls; the decode warps and the x warp wait on the MMA
// completion of the buffer they refill themselves, so that the MMA warp's
// loop is only ready barrier, x wait, MMA issue and commit. A waiter cannot
// fall two phases behind on such a barrier: its next completion needs the
// waiter's own next stage first. Every mbarrier wait is bounded: on a
// timeout the kernel records an error and from then on skips all work while
// still taking every named barrier, so each warp reaches the end and TMEM is
// released.
#pragma once
#include "exl3_kernels.cuh"

namespace tfx {

constexpr int kTcRowsMax = 128;   // rows per pass (MMA N) when a call has at most this many rows
constexpr int kTcRowsLong = 64;   // rows per pass above that (keeps all C chunks in one CTA)
constexpr int kTcSK = 8;          // k-steps per stage
constexpr int kTcDecodeWarps = 16;
constexpr int kTcFoldWarp0 = 16;  // 4 fold warps; TMEM lane quarter = warp % 4
constexpr int kTcMmaWarp = 20;
constexpr int kTcXWarp = 21;
constexpr int kTcThreads = 22 * 32;
constexpr int kTcXS = 3;                              // x ring stages
constexpr int kTcXLanes = 4;                          // lanes that copy a stage's x (one slice each)
constexpr int kTcXStage = kTcSK * kTcRowsMax * 32;    // x bytes per stage (32 KB)
constexpr int kTcAB = 3;                              // A (decoded weight) buffers
constexpr int kTcAStage = kTcSK * 128 * 32;           // A bytes per stage (32 KB)
constexpr int kTcExBytes = 2 * 4 * 128 * 4;           // epilogue exchange (two 4-row groups)
constexpr size_t kTcDynSmem = (size_t)kTcXS * kTcXStage + kTcAB * kTcAStage + kTcExBytes;
// named barriers (0 is __syncthreads)
constexpr int kBarFold = 1;        // the 4 fold warps
constexpr int kBarReady = 2;       // + A buffer: decode warps -> MMA warp (3 ids)
constexpr int kBarFolded = 5;      // + chunk parity: fold warps -> MMA warp (2 ids)
constexpr int kReadyThreads = (kTcDecodeWarps + 1) * 32;
constexpr int kFoldedThreads = 5 * 32;

// Wait for the phase of the given parity to complete, at most `spin` cycles.
// The thread polls with the non-blocking test (a try_wait on an incomplete
// phase suspends the thread for a fixed slice instead of until completion),
// sleeping sleep_ns between polls so that waiting warps leave the issue slots
// of their scheduler to the warps doing work.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err,
                                          long long spin, int sleep_ns = 0) {
  if (*abort_flag) return false;
  if (mbar_poll(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_poll(b, parity)) {
    if (*abort_flag) return false;
    if (sleep_ns) __nanosleep(sleep_ns);
    if (clock64() - t0 > spin) {
      *abort_flag = 1;
      atomicExch(err, 1);
      return false;
    }
  }
  return true;
}
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

constexpr int kTcMaxLevels = 4;  // chunk tree levels parked in TMEM (C <= 16)

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes (one round trip).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Rotated x in the tensor-core layout. Rows are cut into passes of RP rows;
// pass p holds NMp = min(RP, rows_pad - p*RP) rows (a multiple of 16) and its
// element (r', k) sits at byte p*RP*K*2 + tk*NMp*32 + ((r'/8)*2 + (k%16)/8)*128
// + (r'%8)*16 + (k%8)*2, so the rows of a pass at consecutive k-steps are one
// contiguous run that a single bulk copy moves.
__host__ __device__ __forceinline__ long long xc_byte(int r, int k, int K, int RP, int rows_pad) {
  const int p = r / RP, rr = r - p * RP;
  const int NMp = rows_pad - p * RP < RP ? rows_pad - p * RP : RP;
  const int tk = k >> 4, kk = k & 15;
  return (long long)p * RP * K * 2 + (long long)tk * NMp * 32 + ((rr >> 3) * 2 + (kk >> 3)) * 128 + (rr & 7) * 16 +
         (kk & 7) * 2;
}

struct TcArgs {
  LinearArgs la;   // la.m[i].cta_begin is the member's first unit; la.rp the slab row stride
  int units;       // work units of all members
  int RP;          // rows per pass
  int NMf;         // TMEM columns per region: min(RP, rows_pad)
  int* err;        // device error word: 1 when a wait timed out, 2 on a short shared-memory launch
};

struct TcUnit {
  int mi, pass, gidx, nb;
  int tbeg, nsteps;  // first k-step and k-steps of the unit's chunks
  int row0, prow, NMp;
};

__device__ __forceinline__ TcUnit tc_unit(const TcArgs& ta, int u) {
  const LinearArgs& a = ta.la;
  TcUnit U;
  U.mi = 0;
  if (a.count > 1 && u >= a.m[1].cta_begin) U.mi = 1;
  if (a.count > 2 && u >= a.m[2].cta_begin) U.mi = 2;
  const Member& M = a.m[U.mi];
  int local = u - M.cta_begin;
  U.gidx = local % M.P;
  local /= M.P;
  U.nb = local % M.NB;
  U.pass = local / M.NB;
  const int c0 = U.gidx * M.G;
  U.tbeg = chunk_begin(c0, a.TK, M.C);
  U.nsteps = chunk_begin(c0 + M.G, a.TK, M.C) - U.tbeg;
  U.row0 = U.pass * ta.RP;
  U.prow = min(ta.RP, a.rows - U.row0);
  U.NMp = (U.prow + 15) & ~15;
  return U;
}

__device__ __forceinline__ void fold_bar() { bar_sync(kBarFold, 128); }
// All 128 fold threads agree: true only if every one passed ok.
__device__ __forceinline__ bool fold_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.and.pred q, 1, 128, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}
// One lane polls, the warp follows with a warp-uniform outcome.
__device__ __forceinline__ bool wait_lane0(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err,
                                           long long spin, int lane, int sleep_ns) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(b, parity, abort_flag, err, spin, sleep_ns);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Rows r0..r0+3 of one 128-column block, thread = column n = 32*(warp%4) + lane
// of the four fold warps: finish the Walsh-Hadamard transform over n in the
// same stage order as fwht128 (n bits 0..4 across lanes, then bits 5 and 6
// through shared memory), scale by 1/sqrt(128) and svh, store y.
__device__ __forceinline__ void tc_rot_out_store(float (&v)[4], int n, int lane, float* ex, float sv, const Member& M,
                                                 long long row0, int ncol, int nrows, int act) {
#pragma unroll
  for (int m = 0; m < 5; m++) {
    const bool hi = (lane >> m) & 1;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const float o = __shfl_xor_sync(0xffffffffu, v[e], 1 << m);
      v[e] = hi ? (o - v[e]) : (v[e] + o);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; e++) ex[e * 128 + n] = v[e];
  fold_bar();
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const float a5 = ex[e * 128 + (n ^ 32)], b = ex[e * 128 + (n ^ 64)], c = ex[e * 128 + (n ^ 96)];
    const bool h5 = n & 32;
    const float u0 = h5 ? (a5 - v[e]) : (v[e] + a5);
    const float u1 = h5 ? (c - b) : (b + c);
    float o = (n & 64) ? (u1 - u0) : (u0 + u1);
    o = (o * kInvSqrt128) * sv;
    if (e < nrows) store_y1(M, act, row0 + e, ncol, o);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kTcThreads, 1) linear_tc_kernel(const __grid_constant__ TcArgs ta) {
  using WF = WordFetch<BITS>;
  constexpr int kH = kTcSK / 2;  // tiles per decode warp per stage
  const LinearArgs& a = ta.la;
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sX = dsm;                                  // [kTcXS][kTcXStage]
  unsigned char* sA = sX + kTcXS * kTcXStage;               // [kTcAB][kTcAStage]
  float* sEx = reinterpret_cast<float*>(sA + kTcAB * kTcAStage);  // [2][4][128]
  static_assert(kTcAB == kTcXS, "one commit per stage frees its A buffer and its x slot");
  __shared__ __align__(8) uint64_t xfull[kTcXS], sdone[kTcAB], chunk_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  griddep_wait();
  griddep_launch();
  {
    // the launch must provide the shared memory the kernel lays out
    uint32_t dyn;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (dyn < kTcDynSmem) {
      if (threadIdx.x == 0) atomicExch(ta.err, 2);
      return;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // TMEM: two accumulator regions plus log2(G) parked tree levels of NMf columns
  int maxlog = a.m[0].log2G;
  for (int i = 1; i < a.count; i++) maxlog = max(maxlog, a.m[i].log2G);
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)((2 + maxlog) * ta.NMf)) tmem_cols *= 2;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kTcXS; i++) {
      mbar_init(&xfull[i], 1);
    }
    for (int i = 0; i < kTcAB; i++) mbar_init(&sdone[i], 1);
    for (int i = 0; i < 2; i++) mbar_init(&chunk_done[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(&s_tmem)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int NMf = ta.NMf;

  if (warp < kTcDecodeWarps) {
    // ---------------- decode: tile column j, k-steps q0 .. q0+kH-1 of every stage
    const int j = warp & 7, q0 = (warp >> 3) * kH;
    LaneWindow<BITS> lw;
    lw.init(lane);
    const int g = lane >> 2, t = lane & 3;
    const int off0 = 512 * j + 16 * g + 4 * t;  // A-fragment register 0 in the core-matrix layout
    // the words of stage gs sit in register slot gs % NS; the slot of the
    // stage just decoded is refilled with the words NS-1 stages ahead, so a
    // load has NS-1 stages of decode to land (the loop is unrolled NS times
    // so that every slot is a fixed set of registers: no in-flight load is
    // ever copied)
    constexpr int NS = WF::kOwn <= 2 ? 3 : 2;
    uint32_t own[NS][kH][WF::kOwn];
    auto load_stage = [&](const TcUnit& U, int s0, uint32_t (&dst)[kH][WF::kOwn]) {
      const Member& M = a.m[U.mi];
      const uint32_t* col = M.trellis + (long long)(U.nb * 8 + j) * (8 * BITS);
#pragma unroll
      for (int h = 0; h < kH; h++)
        if (s0 + q0 + h < U.nsteps) WF::load(col + (long long)(U.tbeg + s0 + q0 + h) * M.stride, lw, lane, dst[h]);
    };
    // stage iterators: (u, s0, U) the stage to decode, (lu, ls0, LU) the next one to load
    int u = blockIdx.x, s0 = 0, gs = 0;
    TcUnit U;
    if (u < ta.units) U = tc_unit(ta, u);
    int lu = u, ls0 = 0;
    TcUnit LU = U;
    auto advance = [&](int& uu, int& ss, TcUnit& UU) {
      ss += kTcSK;
      if (ss >= UU.nsteps) {
        uu += gridDim.x;
        ss = 0;
        if (uu < ta.units) UU = tc_unit(ta, uu);
      }
    };
#pragma unroll
    for (int sl = 0; sl < NS - 1; sl++) {
      if (lu < ta.units) {
        load_stage(LU, ls0, own[sl]);
        advance(lu, ls0, LU);
      }
    }
    while (u < ta.units) {
#pragma unroll
      for (int sl = 0; sl < NS; sl++) {
        if (u < ta.units) {
          // refill the slot decoded last (stage gs-1) with stage gs+NS-1
          if (lu < ta.units) {
            load_stage(LU, ls0, own[(sl + NS - 1) % NS]);
            advance(lu, ls0, LU);
          }
          const int cnt = min(kTcSK, U.nsteps - s0);
          const int ab = gs % kTcAB;
          // buffer ab last held stage gs - kTcAB: wait until its MMAs completed
          if (gs >= kTcAB) {
            if (lane == 0) mbar_wait(&sdone[ab], ((gs - kTcAB) / kTcAB) & 1, &s_abort, ta.err, a.spin);
            __syncwarp();
          }
          if (!s_abort) {
            unsigned char* abuf = sA + ab * kTcAStage;
#pragma unroll
            for (int h = 0; h < kH; h++) {
              if (q0 + h < cnt) {
                uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
                WF::gather(own[sl][h], lw, lane, raw);
                lw.align(raw, win);
                decode8<BITS>(win, af);
                unsigned char* o = abuf + (q0 + h) * 4096 + off0;
                *reinterpret_cast<uint32_t*>(o) = af[0];        // n = g,   k = 2t..
                *reinterpret_cast<uint32_t*>(o + 256) = af[1];  // n = g+8, k = 2t..
                *reinterpret_cast<uint32_t*>(o + 128) = af[2];  // n = g,   k = 2t+8..
                *reinterpret_cast<uint32_t*>(o + 384) = af[3];  // n = g+8, k = 2t+8..
              }
            }
            fence_async_smem();
          }
          bar_arrive(kBarReady + ab, kReadyThreads);
          gs++;
          advance(u, s0, U);
        }
      }
    }
  } else if (warp < kTcFoldWarp0 + 4) {
    // ---------------- fold and output: thread = TMEM lane = column n of the block
    const int lg = warp & 3, n = 32 * lg + lane;
    const uint32_t lane_base = (uint32_t)(lg * 32) << 16;
    int gc = -1, exb = 0;
    for (int u = blockIdx.x; u < ta.units; u += gridDim.x) {
      const TcUnit U = tc_unit(ta, u);
      const Member& M = a.m[U.mi];
      const float sv = __half2float(M.svh[U.nb * 128 + n]);
      const long long slab = (long long)a.rp * M.N;
      for (int c = 0; c < M.G; c++) {
        gc++;
        const bool ok = fold_all(wait_lane0(&chunk_done[gc & 1], (gc >> 1) & 1, &s_abort, ta.err, a.spin, lane, 64));
        if (ok) {
          tc_fence_after();
          const uint32_t cur = tmem + lane_base + (uint32_t)((gc & 1) * NMf);
          const bool final = c + 1 == M.G;
          // 16 columns (rows of the pass) at a time: cur + the levels the tree
          // prescribes, parked again or written out
          for (int cc = 0; cc < U.NMp; cc += 16) {
            float v[16];
            tmem_ld16(cur + (uint32_t)cc, v);
            int l = 0;
            for (; l < kTcMaxLevels && ((c >> l) & 1); l++) {
              float w[16];
              tmem_ld16(tmem + lane_base + (uint32_t)((2 + l) * NMf + cc), w);
#pragma unroll
              for (int e = 0; e < 16; e++) v[e] = w[e] + v[e];
            }
            if (!final) {
              tmem_st16(tmem + lane_base + (uint32_t)((2 + l) * NMf + cc), v);
            } else if (M.P == 1) {
#pragma unroll
              for (int q = 0; q < 4; q++) {
                float v4[4] = {v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]};
                tc_rot_out_store(v4, n, lane, sEx + (exb & 1) * 512, sv, M, U.row0 + cc + 4 * q, U.nb * 128 + n,
                                 U.prow - cc - 4 * q, a.act);
                exb++;
              }
            } else {
              float* part =
                  M.partial + ((long long)U.pass * M.P + U.gidx) * slab + (long long)cc * M.N + U.nb * 128 + n;
#pragma unroll
              for (int e = 0; e < 16; e++)
                if (cc + e < U.prow) part[(long long)e * M.N] = v[e];
            }
          }
          tc_fence_before();
        }
        bar_arrive(kBarFolded + (gc & 1), kFoldedThreads);
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ---------------- MMA issue, strictly in k order; lane 0 issues, the warp takes the barriers
    const uint64_t da0 = umma_desc(sA), db0 = umma_desc(sX);
    int gs = 0, gc = -1;
    for (int u = blockIdx.x; u < ta.units; u += gridDim.x) {
      const TcUnit U = tc_unit(ta, u);
      const Member& M = a.m[U.mi];
      const uint32_t idesc = umma_idesc(U.NMp);
      const int log2C = __ffs(M.C) - 1;
      const int c0 = U.gidx * M.G;
      int ci = -1, cnext = 0;
      uint32_t acc = 0, dcol = 0;
      for (int s0 = 0; s0 < U.nsteps; s0 += kTcSK, gs++) {
        const int cnt = min(kTcSK, U.nsteps - s0);
        const int ab = gs % kTcAB, xs = gs % kTcXS;
        bar_sync(kBarReady + ab, kReadyThreads);
        int okx = 1;
        if (lane == 0) okx = mbar_wait(&xfull[xs], (gs / kTcXS) & 1, &s_abort, ta.err, a.spin);
        okx = __shfl_sync(0xffffffffu, okx, 0);
        tc_fence_after();
        const bool go = okx && !s_abort;
        const uint64_t da = da0 + (uint64_t)((ab * kTcAStage) >> 4);
        const uint64_t db = db0 + (uint64_t)((xs * kTcXStage) >> 4);
        const uint32_t db_step = (uint32_t)(U.NMp * 32) >> 4;
        // the stage's k-steps as runs inside one chunk: a chunk start first
        // resets the accumulator (and waits until its TMEM region was folded),
        // then lane 0 issues the run back to back and, if the run ends the
        // chunk, commits it to the fold warps
        for (int q = 0; q < cnt;) {
          if (s0 + q == cnext) {
            ci++;
            gc++;
            acc = 0;
            dcol = (uint32_t)((gc & 1) * NMf);
            cnext = (int)(((long long)(c0 + ci + 1) * a.TK) >> log2C) - U.tbeg;  // chunk_begin, C a power of two
            // the region of chunk gc last held chunk gc-2: it must have been folded
            if (gc >= 2) bar_sync(kBarFolded + (gc & 1), kFoldedThreads);
            tc_fence_after();
          }
          const int qe = min(cnt, cnext - s0);
          if (lane == 0) {
            if (go)
              for (int i = q; i < qe; i++) {
                umma_f16(tmem + dcol, da + (uint64_t)(i * (4096 >> 4)), db + (uint64_t)(i * db_step), idesc, acc);
                acc = 1;
              }
            if (s0 + qe == cnext) umma_commit(&chunk_done[gc & 1]);
          }
          acc = 1;
          q = qe;
        }
        // frees A buffer ab and x slot xs (the same index): the decode warps
        // and the x warp wait on it themselves
        if (lane == 0) umma_commit(&sdone[ab]);
        __syncwarp();
      }
    }
    // the folds of the last two chunks
    for (int c = gc - 1; c <= gc; c++)
      if (c >= 0) bar_sync(kBarFolded + (c & 1), kFoldedThreads);
  } else {
    // ---------------- x rows of the pass: one contiguous run per stage, cut
    // into kTcXLanes slices that as many lanes copy: the bulk copies of one
    // thread complete one after another (measured on GB300: about one per
    // 0.45 us whatever their size up to 64 KB), those of different threads overlap
    if (lane < kTcXLanes) {
      constexpr unsigned kMask = (1u << kTcXLanes) - 1;
      int gs = 0;
      for (int u = blockIdx.x; u < ta.units; u += gridDim.x) {
        const TcUnit U = tc_unit(ta, u);
        const Member& M = a.m[U.mi];
        const unsigned char* xsrc =
            reinterpret_cast<const unsigned char*>(M.xf) + (long long)U.pass * ta.RP * a.K * 2;
        for (int s0 = 0; s0 < U.nsteps; s0 += kTcSK, gs++) {
          const int cnt = min(kTcSK, U.nsteps - s0);
          const int xs = gs % kTcXS;
          int ok = 1;
          if (lane == 0 && gs >= kTcXS) ok = mbar_wait(&sdone[xs], ((gs - kTcXS) / kTcXS) & 1, &s_abort, ta.err, a.spin, 32);
          ok = __shfl_sync(kMask, ok, 0);
          if (!ok || s_abort) continue;
          // bytes = cnt * NMp * 32 is a multiple of 512: every slice is a multiple of 16 bytes
          const uint32_t bytes = (uint32_t)(cnt * U.NMp * 32), slice = bytes / kTcXLanes;
          if (lane == 0) mbar_expect_tx(&xfull[xs], bytes);
          __syncwarp(kMask);
          bulk_g2s(sX + xs * kTcXStage + lane * slice,
                   xsrc + (long long)(U.tbeg + s0) * U.NMp * 32 + (long long)lane * slice, slice, &xfull[xs]);
        }
      }
      if (s_abort) {
        // let copies already in flight land before the CTA's shared memory goes away
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

// Split-K combine of the tensor-core kernel's slabs when a block has P > 1
// chunk groups: one warp per (pass, row, 128-column block) folds the P slabs
// as a tree, rotates back (FWHT, 1/sqrt(128)), scales by svh and stores y:
// the same arithmetic, in the same order, as block_epilogue.
struct CombineArgs {
  LinearArgs la;
  int RP;
  long long items[3];  // warps of each member (rows * NB); prefix over members
};

// tc_combine_kernel (defined once, in exl3_host.cu).

}  // namespace tfx
