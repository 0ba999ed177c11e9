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
// (member, pass, 128-column block, chunk group) in a fixed stride. A unit's
// chunks go in pairs (2p, 2p+1) whose two MMA chains are issued alternately,
// each into its own accumulator region: an MMA into the accumulator the
// previous MMA wrote waits for it (measured on GB300: about 180 cycles per
// dependent tcgen05.mma whatever N, about 90 when two chains alternate), and
// the pair's sum is the chunk tree's first level, so the bits do not change.
// The work of a pair is cut into stages of kTcHalf k-steps of each chunk
// (kTcSK = 2 kTcHalf slots) that flow through warp roles:
//   warp 14       asks the tensor copy engine for each stage's trellis words
//                 (2-D boxes of 4 tile rows x 4 tiles, one per lane 0..3: the
//                 first chunk's rows, then the second's) into
//                 a ring of tc_word_stages(BITS) stages, as far ahead as the
//                 ring allows;
//   warp 13       bulk-copies the x rows of each stage (two runs, one per
//                 chunk, two lanes each);
//   warps 0..7    decode: warp j turns tile column j of each stage (8 tiles)
//                 into FP16 A operands;
//   warp 12       issues the MMAs, each chain strictly in k order (lane 0);
//   warps 8..11   fold: add each finished pair and merge it into the chunk tree and
//                 write the unit's FP32 subtree sum (the whole z of the block
//                 when the unit covers all C chunks) to its slab;
//                 tc_combine_kernel then folds each block's slabs, rotates back
//                 and stores y, one warp per (row, block), all in parallel.
//                 Measured on GB300 with timestamps inside the kernel: the
//                 rot_out epilogue run by the four fold warps at the end of a
//                 128-row unit took about 54,000 cycles (a third of the unit),
//                 and the pages' split-K form, where the unit that arrives
//                 last on the block's counter folds the slabs, made small
//                 layers 3x slower (one CTA reading P x rows x 512 B of slabs
//                 one L2 round trip per 4 rows while its pipeline waits).
// Every hand-off is an mbarrier: full/empty rings for words (copy engine ->
// decode warps -> word warp), the stage slots of x and A together (decode
// warps and the x copy -> MMA warp; MMA completion -> decode warps and x
// warp) and the two TMEM accumulator region pairs (MMA completion -> fold
// warps; fold warps -> MMA warp). A waiter never falls two phases behind: the next
// completion of any of these barriers needs the waiter's own next step first.
// Every wait is bounded by the launch's spin limit. On a timeout the kernel
// records device error 1 and every role leaves its loop at its next wait (the
// waits see the abort flag); before the CTA ends, every thread waits about a
// millisecond so that copies and MMAs in flight land, then TMEM is freed.
//
// The chunk tree parks one partial sum per level above the pairs (up to
// log2(16) - 1 = 3). TMEM holds two pairs of accumulator regions plus the
// first `tlev` levels of NMf columns each within its 512 columns; deeper
// levels go to a per-CTA slot of global scratch (L2-resident, written and read
// back by the same thread). That lets one unit hold all C chunks of a 128-row
// pass, so each weight is decoded once per 128 rows.
#pragma once
#include "exl3_kernels.cuh"

namespace tfx {

constexpr int kTcRowsMax = 128;      // rows per pass (MMA N)
constexpr int kTcRowsNoSpill = 64;   // rows per pass above 128 rows when no level scratch is given
constexpr int kTcHalf = 4;           // k-steps of each chunk of a pair per stage
constexpr int kTcSK = 2 * kTcHalf;   // k-step slots per stage
constexpr int kTcDecodeWarps = 8;    // warp j: tile column j, both chunks of the pair
constexpr int kTcFoldWarp0 = 8;      // 4 fold warps; TMEM lane quarter = warp % 4
constexpr int kTcMmaWarp = 12;
constexpr int kTcXWarp = 13;
constexpr int kTcWWarp = 14;
constexpr int kTcThreads = 15 * 32;
// Stages in flight: x slots and A buffers alike, one barrier pair per slot.
// Measured on GB300 against separate x (3) and A (2) rings with their own
// barriers: one wait and one commit fewer per stage for the MMA warp, and the
// shared memory left for a 64 KB word ring (4 stages in flight at 8 bits; a
// third slot with a 32 KB ring was 25 % slower at 6-8 bits).
constexpr int kTcStages = 2;
constexpr int kTcXS = kTcStages;                      // x ring stages
constexpr int kTcXLanes = 4;                          // lanes that copy a stage's x (one slice each)
constexpr int kTcXStage = kTcSK * kTcRowsMax * 32;    // x bytes per stage (32 KB)
constexpr int kTcAB = kTcStages;                      // A (decoded weight) buffers
constexpr int kTcAStage = kTcSK * 128 * 32;           // A bytes per stage (32 KB)
constexpr int kTcWRing = 64 * 1024;                   // trellis-word ring
constexpr int kTcBoxRows = 4;                         // tile rows per word box
constexpr int kTcMaxLevels = 3;                       // chunk tree levels above the pairs (C <= 16)
constexpr int kTcSpillLevels = 3;                     // levels a CTA may park in global scratch
constexpr size_t kTcDynSmem = (size_t)kTcXS * kTcXStage + kTcAB * kTcAStage + kTcWRing;
constexpr int kBarFold = 1;  // named barrier of the 4 fold warps (0 is __syncthreads)

// Trellis words of one stage (kTcSK tile rows of a 128-column block) and how
// many stages the ring holds (at most 8).
__host__ __device__ constexpr int tc_word_stage_bytes(int bits) { return kTcSK * 64 * bits * 4; }
__host__ __device__ constexpr int tc_word_stages(int bits) {
  return kTcWRing / tc_word_stage_bytes(bits) > 8 ? 8 : kTcWRing / tc_word_stage_bytes(bits);
}
// One word box: kTcBoxRows tile rows x 4 tiles (half a block), 32*bits words per row.
__host__ __device__ constexpr int tc_word_box_words(int bits) { return 32 * bits; }
__host__ __device__ constexpr int tc_word_box_bytes(int bits) { return kTcBoxRows * 32 * bits * 4; }

// Wait for the phase of the given parity to complete, at most `spin` cycles;
// gives up at once when the CTA has aborted. On its own timeout it aborts the
// CTA and records device error 1. After one non-blocking test, the thread
// waits with try_wait and a suspend-time hint: it is parked (it issues no
// instructions) until the phase completes or the hint runs out, so waiting
// warps leave the issue slots of their scheduler to the decode warps. (A
// spinning test_wait loop in the MMA warp alone issued about half of the
// kernel's instructions, measured with ncu on GB300.)
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag, int* err,
                                          long long spin) {
  if (mbar_poll(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (clock64() - t0 > spin) {
      *abort_flag = 1;
      atomicExch(err, 1);
      return false;
    }
    if (mbar_test_sleep(b, parity, 20000u)) return true;
  }
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

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// 16 consecutive TMEM columns of this warp's 32 lanes, without waiting: the
// registers are valid after tmem_wait_ld (several loads share one round trip).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 consecutive TMEM columns stored without waiting (tmem_wait_st before the
// columns are read again or handed to another thread).
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
  LinearArgs la;  // la.m[i].cta_begin is the member's first unit; la.rp the slab row stride;
                  // la.tm[i] member i's trellis words, boxes of 4 tiles x kTcBoxRows tile rows
  int units;      // work units of all members
  int RP;         // rows per pass
  int NMf;        // TMEM columns per region: min(RP, rows_pad)
  int tlev;       // chunk tree levels above the pairs parked in TMEM; deeper ones go to `lev`
  int* err;       // device error word: 1 when a wait timed out, 2 on a short shared-memory launch
  float* lev;     // global scratch for deeper levels: per CTA, kTcSpillLevels x NMf x 128 FP32
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
  U.gidx = local & (M.P - 1);  // P is a power of two
  local >>= ilog2_pow2(M.P);
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

// Chunk pair pp of a unit: chunks c = 2pp, 2pp+1 of its group, first k-steps
// ta, tb and lengths na, nb (each at least 4), ns stages of kTcHalf k-steps of each.
struct TcPair {
  int ta, na, tb, nb, ns;
};
__device__ __forceinline__ TcPair tc_pair(const TcArgs& ta_, const Member& M, const TcUnit& U, int pp) {
  const LinearArgs& a = ta_.la;
  const int c = U.gidx * M.G + 2 * pp;
  TcPair P;
  P.ta = chunk_begin(c, a.TK, M.C);
  P.tb = chunk_begin(c + 1, a.TK, M.C);
  const int te = chunk_begin(c + 2, a.TK, M.C);
  P.na = P.tb - P.ta;
  P.nb = te - P.tb;
  P.ns = (max(P.na, P.nb) + kTcHalf - 1) / kTcHalf;
  return P;
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
                                           long long spin, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(b, parity, abort_flag, err, spin);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

template <int BITS>
__global__ void __launch_bounds__(kTcThreads, 1) linear_tc_kernel(const __grid_constant__ TcArgs ta) {
  // tiles per decode warp per stage: one decode warp per tile column, two per
  // SM sub-partition. Measured on GB300: with 16 decode warps (4 per
  // sub-partition, 4 tiles each) the single-lane MMA warp, which shares a
  // sub-partition with always-ready decode warps, took about 770 cycles per
  // stage for its loop with no MMA issued; 8 decode warps made gate+up at 128
  // rows 139.5 -> 128.7 us and the 4096-row gate chunk 1880 -> 1717 us (with
  // chunk pairs, 16 warps one per tile column and chunk: 127.6 -> 145.9 us and
  // 1668 -> 1889 us).
  constexpr int kH = kTcSK * 8 / kTcDecodeWarps;  // slots per decode warp per stage
  constexpr int WS = tc_word_stages(BITS);
  constexpr int WSB = tc_word_stage_bytes(BITS);
  constexpr int BOXB = tc_word_box_bytes(BITS);
  const LinearArgs& a = ta.la;
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char* sX = dsm;                               // [kTcXS][kTcXStage]
  unsigned char* sA = sX + kTcXS * kTcXStage;            // [kTcAB][kTcAStage]
  unsigned char* sW = sA + kTcAB * kTcAStage;            // [WS][WSB]
  // sfull[i]: stage slot i holds its decoded A (8 decode-warp arrivals) and
  // its x (the x warp's arrival with the bytes); sdone[i]: the slot's MMAs
  // have completed (one commit frees both the A buffer and the x slot)
  __shared__ __align__(8) uint64_t sfull[kTcStages], sdone[kTcStages], wfull[8], wempty[8],
      cdone[2], tfree[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  griddep_wait();
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
  const long long spin = a.spin;
  // TMEM: two pairs of accumulator regions plus the parked tree levels kept
  // in TMEM (log2(G) - 1 levels above the pairs)
  int maxlog = a.m[0].log2G;
  for (int i = 1; i < a.count; i++) maxlog = max(maxlog, a.m[i].log2G);
  const int maxlev = maxlog - 1;
  if (maxlev < 0 || (4 + min(maxlev, ta.tlev)) * ta.NMf > 512) {
    if (threadIdx.x == 0) atomicExch(ta.err, 2);
    return;
  }
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)((4 + min(maxlev, ta.tlev)) * ta.NMf)) tmem_cols *= 2;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kTcStages; i++) {
      mbar_init(&sfull[i], kTcDecodeWarps + 1);
      mbar_init(&sdone[i], 1);
    }
    for (int i = 0; i < WS; i++) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], kTcDecodeWarps);
    }
    for (int i = 0; i < 2; i++) {
      mbar_init(&cdone[i], 1);
      mbar_init(&tfree[i], 4);
    }
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
    // ---------------- decode: tile column j, every k-step of every stage
    const int j = warp & 7, q0 = (warp >> 3) * kH;
    LaneWindow<BITS> lw;
    lw.init(lane);
    const int g = lane >> 2, t = lane & 3;
    const int off0 = 512 * j + 16 * g + 4 * t;  // A-fragment register 0 in the core-matrix layout
    // tile (h, j) of a word stage: box (h/4, j/4), row h%4, tile j%4
    const int wofs = (j >> 2) * BOXB + (j & 3) * 32 * BITS;
    int gs = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < ta.units && ok; u += gridDim.x) {
      const TcUnit U = tc_unit(ta, u);
      const Member& M = a.m[U.mi];
      for (int pp = 0; pp < (M.G >> 1) && ok; pp++) {
      const TcPair P = tc_pair(ta, M, U, pp);
      for (int s = 0; s < P.ns; s++, gs++) {
        // slots 0..3: the first chunk's k-steps 4s.., slots 4..7: the second's
        const int ws = gs % WS, ab = gs % kTcAB;
        ok = wait_lane0(&wfull[ws], (uint32_t)(gs / WS) & 1u, &s_abort, ta.err, spin, lane);
        // buffer ab last held stage gs - kTcAB: its MMAs must have completed
        if (ok && gs >= kTcAB)
          ok = wait_lane0(&sdone[ab], (uint32_t)((gs - kTcAB) / kTcAB) & 1u, &s_abort, ta.err, spin, lane);
        if (!ok) break;
        const unsigned char* wst = sW + ws * WSB + wofs;
        unsigned char* abuf = sA + ab * kTcAStage;
        // every slot is decoded and stored, also those past the end of a
        // chunk (stale words of this ring slot into A slots no MMA reads):
        // straight-line code lets the compiler interleave the 8 tiles, which
        // two decode warps per SM sub-partition need to hide latency (measured
        // on GB300: gate+up at 64 rows 108.6 -> 95.1 us, the 4096-row gate
        // chunk 1671 -> 1519 us, against a guard per slot)
#pragma unroll
        for (int h = 0; h < kH; h++) {
          {
            const int hh = q0 + h;
            const uint32_t* tile = reinterpret_cast<const uint32_t*>(wst + (hh >> 2) * 2 * BOXB + (hh & 3) * 128 * BITS);
            uint32_t raw[Geo<BITS>::kRaw], win[Geo<BITS>::kNorm + 1], af[4];
            raw[0] = tile[lw.i0];
            raw[1] = tile[lw.i1];
            if constexpr (Geo<BITS>::kRaw > 2) raw[2] = tile[lw.i2];
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
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sfull[ab]);
          mbar_arrive(&wempty[ws]);
        }
      }
      }
    }
  } else if (warp < kTcFoldWarp0 + 4) {
    // ---------------- fold and output: thread = TMEM lane = column n of the block
    const int lg = warp & 3, n = 32 * lg + lane;
    const uint32_t lane_base = (uint32_t)(lg * 32) << 16;
    float* spill = ta.lev ? ta.lev + (size_t)blockIdx.x * kTcSpillLevels * NMf * 128 + n : nullptr;
    int gc = -1;
    bool ok = true;
    for (int u = blockIdx.x; u < ta.units && ok; u += gridDim.x) {
      const TcUnit U = tc_unit(ta, u);
      const Member& M = a.m[U.mi];
      const long long slab = (long long)a.rp * M.N;
      for (int pp = 0; pp < (M.G >> 1); pp++) {
        gc++;
        ok = fold_all(wait_lane0(&cdone[gc & 1], (uint32_t)(gc >> 1) & 1u, &s_abort, ta.err, spin, lane));
        if (!ok) break;
        tc_fence_after();
        // the pair's two regions: chunk 2pp, then chunk 2pp+1
        const uint32_t cur = tmem + lane_base + (uint32_t)((gc & 1) * 2 * NMf);
        const bool final = pp + 1 == (M.G >> 1);
        // the levels above the pairs this pair closes: pp's trailing one bits
        // (all of them for the unit's last pair), the first `tlev` in TMEM
        int nlev = 0;
        while (nlev < kTcMaxLevels && ((pp >> nlev) & 1)) nlev++;
        const int nt = min(nlev, ta.tlev);
        // 16 columns (rows of the pass) at a time: the pair's sum + the levels
        // the tree prescribes (lowest first), parked again or written out. The
        // TMEM loads of a group share one round trip; stores are not waited
        // for until the pair is done.
        for (int cc = 0; cc < U.NMp; cc += 16) {
          float v[16];
          {
            uint32_t r0[16], r1[16], r2[16];
            tmem_ld16_async(cur + (uint32_t)cc, r0);
            tmem_ld16_async(cur + (uint32_t)(NMf + cc), r1);
            if (nt > 0) tmem_ld16_async(tmem + lane_base + (uint32_t)(4 * NMf + cc), r2);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e++) v[e] = __uint_as_float(r0[e]) + __uint_as_float(r1[e]);
            if (nt > 0)
#pragma unroll
              for (int e = 0; e < 16; e++) v[e] = __uint_as_float(r2[e]) + v[e];
            if (nt > 1) {
              tmem_ld16_async(tmem + lane_base + (uint32_t)(5 * NMf + cc), r1);
              if (nt > 2) tmem_ld16_async(tmem + lane_base + (uint32_t)(6 * NMf + cc), r2);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; e++) v[e] = __uint_as_float(r1[e]) + v[e];
              if (nt > 2)
#pragma unroll
                for (int e = 0; e < 16; e++) v[e] = __uint_as_float(r2[e]) + v[e];
            }
            // levels parked in global scratch (only pairs that close a level
            // beyond TMEM's), lowest first
            for (int l = ta.tlev; l < nlev; l++) {
              const float* src = spill + (size_t)((l - ta.tlev) * NMf + cc) * 128;
#pragma unroll
              for (int e = 0; e < 16; e++) v[e] = __ldcg(src + e * 128) + v[e];
            }
          }
          if (!final) {
            // park at level nlev (the first clear bit of pp)
            if (nlev < ta.tlev) {
              tmem_st16_async(tmem + lane_base + (uint32_t)((4 + nlev) * NMf + cc), v);
            } else {
              float* dst = spill + (size_t)((nlev - ta.tlev) * NMf + cc) * 128;
#pragma unroll
              for (int e = 0; e < 16; e++) __stcg(dst + e * 128, v[e]);
            }
          } else {
            float* part = M.partial + ((long long)U.pass * M.P + U.gidx) * slab + (long long)cc * M.N + U.nb * 128 + n;
#pragma unroll
            for (int e = 0; e < 16; e++)
              if (cc + e < U.prow) __stcg(part + (long long)e * M.N, v[e]);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tfree[gc & 1]);
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ---------------- MMA issue by lane 0: per stage the pair's two chains
    // alternately, each strictly in k order
    if (lane == 0) {
      const uint64_t da0 = umma_desc(sA), db0 = umma_desc(sX);
      int gs = 0, gc = -1;
      bool ok = true;
      for (int u = blockIdx.x; u < ta.units && ok; u += gridDim.x) {
        const TcUnit U = tc_unit(ta, u);
        const Member& M = a.m[U.mi];
        const uint32_t idesc = umma_idesc(U.NMp);
        const uint32_t db_step = (uint32_t)(U.NMp * 32) >> 4;
        for (int pp = 0; pp < (M.G >> 1) && ok; pp++) {
          const TcPair P = tc_pair(ta, M, U, pp);
          gc++;
          const uint32_t d0 = tmem + (uint32_t)((gc & 1) * 2 * NMf), d1 = d0 + (uint32_t)NMf;
          for (int s = 0; s < P.ns; s++, gs++) {
            const int cnta = min(kTcHalf, P.na - kTcHalf * s), cntb = min(kTcHalf, P.nb - kTcHalf * s);
            const int ab = gs % kTcAB, xs = gs % kTcXS;
            ok = mbar_wait(&sfull[ab], (uint32_t)(gs / kTcStages) & 1u, &s_abort, ta.err, spin);
            // the pair's regions last held pair gc-2: it must have been folded
            if (ok && s == 0 && gc >= 2) ok = mbar_wait(&tfree[gc & 1], (uint32_t)((gc - 2) >> 1) & 1u, &s_abort, ta.err, spin);
            if (!ok) break;
            tc_fence_after();
            const uint64_t da = da0 + (uint64_t)((ab * kTcAStage) >> 4);
            const uint64_t db = db0 + (uint64_t)((xs * kTcXStage) >> 4);
#pragma unroll
            for (int q = 0; q < kTcHalf; q++) {
              const uint32_t acc = (s > 0 || q > 0) ? 1u : 0u;
              if (q < cnta) umma_f16(d0, da + (uint64_t)(q * (4096 >> 4)), db + (uint64_t)(q * db_step), idesc, acc);
              if (q < cntb)
                umma_f16(d1, da + (uint64_t)((kTcHalf + q) * (4096 >> 4)), db + (uint64_t)((kTcHalf + q) * db_step),
                         idesc, acc);
            }
            if (s + 1 == P.ns) umma_commit(&cdone[gc & 1]);
            // frees A buffer and x slot ab once these MMAs have completed
            umma_commit(&sdone[ab]);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kTcXWarp) {
    // ---------------- x rows of the pass: two contiguous runs per stage (one
    // per chunk of the pair), each cut into two slices that as many lanes
    // copy: the bulk copies of one thread complete one after another
    // (measured on GB300: about one per 0.45 us whatever their size up to 64
    // KB), those of different threads overlap
    if (lane < kTcXLanes) {
      constexpr unsigned kMask = (1u << kTcXLanes) - 1;
      int gs = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < ta.units && ok; u += gridDim.x) {
        const TcUnit U = tc_unit(ta, u);
        const Member& M = a.m[U.mi];
        const unsigned char* xsrc =
            reinterpret_cast<const unsigned char*>(M.xf) + (long long)U.pass * ta.RP * a.K * 2;
        for (int pp = 0; pp < (M.G >> 1) && ok; pp++) {
          const TcPair P = tc_pair(ta, M, U, pp);
          for (int s = 0; s < P.ns; s++, gs++) {
            const int cnta = max(0, min(kTcHalf, P.na - kTcHalf * s)), cntb = max(0, min(kTcHalf, P.nb - kTcHalf * s));
            const int xs = gs % kTcXS;
            int okl = 1;
            if (lane == 0 && gs >= kTcXS)
              okl = mbar_wait(&sdone[xs], (uint32_t)((gs - kTcXS) / kTcXS) & 1u, &s_abort, ta.err, spin);
            ok = __shfl_sync(kMask, okl, 0) != 0;
            if (!ok) break;
            // two runs (the first chunk's k-steps to slots 0.., the second's to
            // slots kTcHalf..), each cut in two halves: cnt * NMp * 16 bytes, a
            // multiple of 256
            // the x warp's arrival on the stage's barrier, with the bytes to come
            if (lane == 0) mbar_expect_tx(&sfull[xs], (uint32_t)((cnta + cntb) * U.NMp * 32));
            __syncwarp(kMask);
            const int second = lane >> 1, half = lane & 1;
            const int cnt = second ? cntb : cnta;
            if (cnt > 0) {
              const uint32_t slice = (uint32_t)(cnt * U.NMp * 16);
              const int t0 = (second ? P.tb : P.ta) + kTcHalf * s;
              bulk_g2s(sX + xs * kTcXStage + second * kTcHalf * U.NMp * 32 + half * slice,
                       xsrc + (long long)t0 * U.NMp * 32 + (long long)half * slice, slice, &sfull[xs]);
            }
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- trellis words: per stage, 2-D boxes of 4 tiles x 4 tile
    // rows (two per chunk of the pair) into the ring, one box per lane of
    // lanes 0..3 (copies issued by one thread complete one after another, so
    // a stage's boxes come from four threads); a slot is refilled once every
    // decode warp has consumed it
    if (lane < 4) {
      constexpr unsigned kMask = 0xFu;
      const int rb = lane >> 1, hx = lane & 1;
      int gs = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < ta.units && ok; u += gridDim.x) {
        const TcUnit U = tc_unit(ta, u);
        const CUtensorMap* tm = &a.tm[U.mi];
        const Member& M = a.m[U.mi];
        for (int pp = 0; pp < (M.G >> 1) && ok; pp++) {
          const TcPair P = tc_pair(ta, M, U, pp);
          for (int s = 0; s < P.ns; s++, gs++) {
            const bool va = P.na > kTcHalf * s, vb = P.nb > kTcHalf * s;
            const int ws = gs % WS;
            int okl = 1;
            if (lane == 0 && gs >= WS) okl = mbar_wait(&wempty[ws], (uint32_t)((gs - WS) / WS) & 1u, &s_abort, ta.err, spin);
            ok = __shfl_sync(kMask, okl, 0) != 0;
            if (!ok) break;
            // box row 0: the first chunk's tile rows ta + 4s.., box row 1: the second's
            if (lane == 0) mbar_expect_tx(&wfull[ws], (uint32_t)(((va ? 1 : 0) + (vb ? 1 : 0)) * 2 * BOXB));
            __syncwarp(kMask);
            if (rb == 0 ? va : vb)
              tma_load_2d(sW + ws * WSB + (rb * 2 + hx) * BOXB, tm, (U.nb * 8 + hx * 4) * 8 * BITS,
                          (rb == 0 ? P.ta : P.tb) + kTcHalf * s, &wfull[ws]);
          }
        }
      }
    }
    __syncwarp();
  }
  // with programmatic dependent launch, the next kernel may start launching
  // once every CTA has finished its units (its CTAs wait for this grid before
  // they read its output)
  griddep_launch();
  if (s_abort) {
    // a wait gave up: let copies and MMAs already in flight land before the
    // CTA's shared memory and tensor memory go away
    const long long t0 = clock64();
    while (clock64() - t0 < 2000000) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

// Split-K combine of the tensor-core kernel's slabs when a block has P > 1
// chunk groups: one warp per (row, 128-column block) folds the P slabs as a
// tree, rotates back (FWHT, 1/sqrt(128)), scales by svh and stores y: the same
// arithmetic, in the same order, as block_epilogue.
struct CombineArgs {
  LinearArgs la;
  int RP;
  long long items[3];  // warps of each member (rows * NB); prefix over members
};

// tc_combine_kernel (defined once, in exl3_host.cu).

}  // namespace tfx
