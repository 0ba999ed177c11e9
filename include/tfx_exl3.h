/*
 * tfx_exl3 — EXL3 trellis-quantized, Hadamard-rotated linear layer for GB300 (sm_103a).
 *
 * C ABI. Every pointer to tensor data is a CUDA device pointer owned by the
 * caller unless stated otherwise; the library never frees caller memory.
 * Every call returns 0 on success or a negative TFX_E* code, never aborts,
 * and on a validation error enqueues nothing. tfx_exl3_last_error() gives a
 * thread-local message for the last failing call.
 *
 * The layer (TensorFold PR #1467 "exl3 cuda: the 27B's EXL3 speed series on
 * the native Dense module", sections "What this changes" and "The arithmetic";
 * PR #1407 item 2):
 *     y = svh o Hn( fp16( Hn(suh o x) ) . W ),   Hn = H128 / sqrt(128) per 128-block
 * where W (K x N) is decoded on the fly from `bits`-per-weight trellis codes
 * stored in 16x16 tiles of 8*bits uint32 words, and the product is summed in
 * FP32 with a deterministic split-K whose per-block arrival counters are reset
 * by the last-arriving CTA (PR #1475 "exl3: zero the split-K counters once as
 * they grow, not before every call", section "What this changes").
 *
 * Decode rule, tile layout and summation order: see the header comment of the
 * kernels (exl3_trellis_quantized_rot_gb300/csrc/exl3_kernels.cuh).
 */
#ifndef TFX_EXL3_H
#define TFX_EXL3_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define TFX_OK 0
#define TFX_EINVAL -1        /* bad argument: shape, bits, count, null pointer */
#define TFX_ENOTRESERVED -2  /* rows above the reserved capacity, or no reserve() yet */
#define TFX_EUNSUPPORTED -3  /* valid but not served (e.g. group members of unequal K) */
#define TFX_EALIGN -4        /* a pointer (or the tile-row stride) is not 16-byte aligned */
#define TFX_ECUDA -5         /* a CUDA runtime call failed; see tfx_exl3_last_error() */

typedef enum { TFX_F16 = 0, TFX_BF16 = 1 } tfx_dtype;

/* A quantized weight. All pointers are caller-owned device memory.
 * trellis : tiles of 8*bits uint32 words; tile (tk, tn) starts at word
 *           tk*tile_row_stride + tn*8*bits, tk < K/16, tn < N/16. The 8 tiles
 *           tn = 8*nb .. 8*nb+7 form 128-column block nb.
 * suh     : K FP16 values (the input sign flips; any FP16 scale is allowed).
 * svh     : N FP16 values (the output sign flips / scales).
 * K, N    : multiples of 128. bits: 1..8.
 * tile_row_stride : words between tile rows; (N/16)*8*bits for a full weight,
 *           the parent's value for a column view. A multiple of 4 words
 *           (TFX_EALIGN otherwise): tile rows are copied as 16-byte runs.
 * act     : dtype of x and y.
 * priv    : library-owned state (scratch, counters), NULL until reserve(). */
typedef struct {
  const uint32_t* trellis;
  const uint16_t* suh;
  const uint16_t* svh;
  int K, N, bits;
  int64_t tile_row_stride;
  int act;
  void* priv;
} tfx_exl3_weight;

/* y[rows x N] = layer(x[rows x K]); x, y row-major in w->act, 16-byte aligned.
 * rows == 0 is a no-op. rows above the reserved max_rows -> TFX_ENOTRESERVED.
 * Enqueued on `stream`; allocates nothing and clears nothing (the counters
 * are reset by the kernel itself). Calls on one weight must be ordered on
 * one stream. Rows are cut into passes (PR #1475, "What this changes":
 * counters indexed pass*NB + nb): one pass up to 128 rows, 64-row passes
 * above that. */
int tfx_exl3_linear(tfx_exl3_weight* w, const void* x, int rows, void* y, cudaStream_t stream);

/* One rotation launch and one linear launch for up to 3 weights of the same
 * K, bits and act over the same rows (PR #1467, "What this changes":
 * matmulGroup runs up to three layers of one K over the same rows in one
 * rotation and one launch). Each member keeps its own suh, svh, plan,
 * scratch and counters; ys[i] is rows x ws[i]->N. Bytes equal those of
 * tfx_exl3_linear on each member. count == 1 is tfx_exl3_linear. */
int tfx_exl3_group(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                   cudaStream_t stream);

/* tfx_exl3_group with an output window per member: member i's output element
 * (r, n) is written at ys[i] + r*ldy[i] + (n - col0[i]) (elements of w->act),
 * for n >= col0[i]; columns below col0[i] are computed but not stored.
 * col0[i]: a multiple of 8 in [0, N); ldy[i]: a multiple of 8, >= N - col0[i].
 * Bytes of every stored element equal those of tfx_exl3_linear on the member.
 * This packs several column views of one weight into one buffer in one call:
 * the drafter's LM head over two vocabulary spans (PR #1507, "What this
 * changes": the head() arm computes the views [0, 98304) and the last 64
 * blocks and packs them into one logits buffer with a 2-D copy that drops the
 * first 7,904 columns of the tail) is group_into over the two views with
 * ldy = 98304 + 288, col0 = {0, 7904}, ys = {logits, logits + 98304}: the
 * epilogue writes the packed layout directly, with no copy. */
int tfx_exl3_group_into(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                        const int64_t ldy[], const int col0[], cudaStream_t stream);

/* One step of a chain: a group call (1..3 members of one K, bits and act)
 * on x, writing ys[i] (rows x ws[i]->N). x is the chain's input or the
 * output of an earlier step (the next layer of the model consumes it). */
typedef struct {
  tfx_exl3_weight* const* ws;
  int count;
  const void* x;
  void* const* ys;
} tfx_exl3_step;

/* Layer-level chaining (PR #1467, "What this changes": the rotations and the
 * decode-row linears chained with programmatic dependent launch so that each
 * launch hides behind the previous one; PR #1475, "What this changes": one
 * reserve at load, so that a captured decode step allocates and clears
 * nothing): the steps' launches are enqueued back to back on `stream`, in
 * order, each step's kernels after the previous step's. pdl selects the
 * programmatic-dependent-launch attribute per launch: 1 on every launch (a
 * kernel may start launching while its predecessor finishes, and waits for
 * it, griddepcontrol.wait, before it reads anything the predecessor wrote or
 * writes anything it reads); 2 the library's automatic choice (that of
 * tfx_exl3_set_pdl mode 2); 0 ordinary stream order. Other values: TFX_EINVAL,
 * nothing enqueued. Every step is validated
 * (shapes, alignment, every member reserved for `rows`) before anything is
 * enqueued; the chain allocates and clears nothing, so it can be captured in
 * a CUDA graph. Bytes equal those of the same group calls made one by one. */
int tfx_exl3_chain(const tfx_exl3_step* steps, int nsteps, int rows, int pdl, cudaStream_t stream);

/* A view of whole 128-column blocks [from, from+n) of w that reads the same
 * stored words and keeps the parent's tile-row stride (PR #1507, "What this
 * changes": exl3.Weight.columns(from, n)). from % 128 == 0, n % 128 == 0,
 * from + n <= w->N. view_out->priv is NULL: reserve the view before use. */
int tfx_exl3_columns(const tfx_exl3_weight* w, int from, int n, tfx_exl3_weight* view_out);

/* tfx_exl3_linear with no allocation at all: the rotated x, split-K partials
 * and counters live in one static device array of 8 MiB built into the
 * library (every GPU that loads the library keeps it until exit) instead of
 * the memory tfx_exl3_reserve obtains. The pages have no counterpart of this
 * call; it serves callers that cannot call cudaMalloc or any other allocator
 * where they run the layer (code running inside a host callback or a context
 * where allocation is forbidden, plugins whose host application owns all
 * device memory, runtimes that must not allocate after start-up).
 * w needs no reserve() (w->priv is ignored); x, y as for tfx_exl3_linear.
 * `stream` must belong to the current device (TFX_EINVAL otherwise).
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture. Each call
 * clears the array's device error word and the counters it uses with one
 * cudaMemsetAsync on `stream` (the array keeps what the previous call left).
 * The device error word cannot be read through tfx_exl3_debug_error (which
 * needs a reserved weight): a static call cannot report a bounded wait that
 * gave up. All calls share the one array: calls that overlap on the GPU race,
 * so order them on one stream. A call whose scratch (counters + rows*K*2 +
 * splits*min(rows,128)*N*4 bytes, rounded) exceeds the array returns
 * TFX_EUNSUPPORTED with the sizes in the message. */
int tfx_exl3_linear_static(const tfx_exl3_weight* w, const void* x, int rows, void* y, cudaStream_t stream);

/* Size the weight's scratch (rotated x, split-K partials, counters) for up
 * to max_rows rows. Grows only; the counter buffer is zeroed on `stream`
 * once per growth and never otherwise (PR #1475, "What this changes").
 * Call before CUDA-graph capture; linear/group then allocate nothing. */
int tfx_exl3_reserve(tfx_exl3_weight* w, int max_rows, cudaStream_t stream);

/* Free priv (synchronises the device first). Safe on an unreserved weight. */
int tfx_exl3_release(tfx_exl3_weight* w);

/* Re-zero the counters on `stream` (recovery after a failed launch). */
int tfx_exl3_reset_counters(tfx_exl3_weight* w, cudaStream_t stream);

/* Write the decoded FP16 weight W (K x N, row-major W[k][n]) to W_out. */
int tfx_exl3_debug_decode(const tfx_exl3_weight* w, uint16_t* W_out, cudaStream_t stream);

/* The summation plan: K is cut into *chunks (a power of two <= 16, at least
 * 4 tiles of 16 rows each, *tiles_per_chunk = (K/16)/chunks rounded down) whose
 * FP32 MMA-chain sums combine by a balanced binary tree in chunk order. A pure
 * function of K: rows, N, views, groups and launch shapes never change it, so
 * a column view always gives the bytes of the same columns of its parent
 * (PR #1507 needed its tail view to take 64 blocks so that plan() gave it the
 * head's K split). */
int tfx_exl3_plan(const tfx_exl3_weight* w, int* chunks, int* tiles_per_chunk);

/* Allocations and counter memsets made for this weight since its creation. */
int tfx_exl3_stats(const tfx_exl3_weight* w, int64_t* allocs, int64_t* memsets);

/* Kernel family for the next calls. 0 = auto: 1..16 rows the warp-granular
 * decode-rows kernel (one cluster of C CTAs per 128-column block folds the C
 * chunk sums in distributed shared memory; launches of more than 128 blocks,
 * or more than 48 blocks at more than 8 rows, write the chunk sums to global
 * slabs that a combine kernel folds instead), every call above 16 rows the
 * tensor-core kernel; 1 = for 1..64 rows the CTA decode-rows kernel whose split-K
 * partials are summed in-kernel by the last CTA to arrive on each block's
 * counter (the counter resets itself); 2 = the tensor-core kernel for every
 * row count; 3 = the warp-granular decode-rows kernel for every call of
 * 1..64 rows (fold chosen as in auto); 4 = as 3, for every call of up to 8
 * rows with the chunk sums folded by the last CTA to arrive on the block's
 * counter (which resets it). Rows a forced family does not serve go to
 * the tensor-core kernel. All give the same bytes. Initial value from
 * TFX_EXL3_VARIANT (auto|rows|mid|warp|warp_global). Returns the previous
 * value; a value outside 0..4 changes nothing. */
int tfx_exl3_set_variant(int variant);

/* Introspection, host only (no GPU needed): the kernel family and tensor-core
 * unit size that a call of `rows` rows over weights of this K and bits, with
 * `blocks` 128-column blocks over all members, would launch under the current
 * variant on a GPU of sm_count SMs (0 = the current device's, 152 when none is
 * visible). *family: 0 = decode-rows CTA kernel (variant rows), 1 = warp-
 * granular decode-rows kernel, 2 = tensor-core kernel. *chunks_per_unit: the
 * chunks of K per tensor-core work unit (G; a launch-shape choice that never
 * changes the bits), 0 for the decode-rows families. TFX_EINVAL on K not a
 * positive multiple of 128, bits outside 1..8, rows or blocks < 1,
 * sm_count < 0 or a null output. */
int tfx_exl3_debug_launch_shape(int K, int bits, int rows, int64_t blocks, int sm_count, int* family,
                                int* chunks_per_unit);

/* Kernels the library has enqueued on any stream (or recorded into a CUDA
 * graph under capture) since it was loaded, counted on the host: the
 * difference across one captured step is the step's launch count. */
int64_t tfx_exl3_debug_launch_count(void);

/* Programmatic dependent launch of the single and group calls (PR #1467,
 * "What this changes"): 0 off, 1 on every launch, 2 automatic (the default:
 * on the rotation launch and the decode-rows linear launch of a call that has
 * both, and on the combine launch that folds a decode-rows launch's slabs;
 * off for fused-rotation and tensor-core launches and the tensor-core
 * combine, the choice that measured fastest inside CUDA graphs). Initial value from TFX_EXL3_PDL
 * ("0" or "1"; unset or anything else: 2). Returns the previous mode, or
 * TFX_EINVAL for a mode outside 0..2 (nothing changed). The static-scratch
 * entry point never uses it. */
int tfx_exl3_set_pdl(int mode);

/* Test hook: replace the allocator and memset used by reserve/release so the
 * host logic runs without a GPU. NULL restores the CUDA runtime. */
typedef struct {
  int (*alloc)(void** p, size_t bytes, cudaStream_t s);
  int (*free)(void* p, cudaStream_t s);
  int (*memset0)(void* p, size_t bytes, cudaStream_t s);
} tfx_exl3_driver;
int tfx_exl3_debug_set_driver(const tfx_exl3_driver* d);

/* Device error word of a reserved weight, written by a launch on it: 1 once
 * a tensor-core launch gave up a bounded wait (its pipeline stopped; the
 * launch skips its remaining work and stores nothing more), 2 if a tensor-core
 * launch got less shared memory than it lays out (it then does nothing), 3
 * once a decode-rows (warp-granular) launch gave up waiting for a copy of
 * trellis words or x into shared memory (its CTA stores nothing), 0
 * otherwise. A wait gives up after the spin limit (about 1 s by default, see
 * tfx_exl3_debug_set_spin_limit); it is never expected on a healthy GPU.
 * Synchronous copy; for tests and diagnostics. reset_counters clears it. */
int tfx_exl3_debug_error(const tfx_exl3_weight* w, int* device_error);

/* Test hook: the clock cycles a bounded wait inside a kernel polls before it
 * gives up (default 2e9, about 1 s); clocks <= 0 restores the default.
 * Applies to launches enqueued after the call. Returns the previous limit.
 * A test lowers it to a few cycles so that waits give up on a healthy GPU and
 * the error path (device error word, reset_counters, a correct next call) can
 * be checked without a fault. */
int64_t tfx_exl3_debug_set_spin_limit(int64_t clocks);

/* Decode-rate probe: launches, on `stream`, the decode rule's arithmetic (one
 * 16x16 tile decode and one m16n8k16 MMA per step, words read from a table in
 * shared memory, no global-memory traffic) at full occupancy, tiles_per_warp
 * tiles per warp, for `bits` 1..8. *weights = weights the launch decodes;
 * *sink_floats = floats `sink` must hold (one per warp). With sink == NULL
 * only the two outputs are set and nothing is launched. The caller times the
 * launch (CUDA events on `stream`): weights / time is the decode rate this GPU
 * sustains for the rule, the ALU roofline of decode-bound calls. */
int tfx_exl3_debug_decode_rate(int bits, int tiles_per_warp, float* sink, int* sink_floats, int64_t* weights,
                               cudaStream_t stream);

/* Synthetic trellis encoder: the tail-biting trellis code of each 16x16 tile
 * whose decoded values are closest (summed squared error) to the targets, by
 * Viterbi search over the bit-shift trellis of the decode rule with QTIP's
 * two-pass tail-biting approximation (Tseng et al., 2024). The pages' weights
 * come from trained checkpoints and show no encoder; this one gives seeded
 * Gaussian weights a real quantize -> decode error per bit width.
 * targets : K x N int16, row-major, device: W[k][n] * 128 rounded to an
 *           integer (the value grid of the decode rule), clamped to
 *           [-1024, 1023] by the kernel.
 * trellis : out, device, the tile layout of tfx_exl3_weight with
 *           tile_row_stride = (N/16)*8*bits; 16-byte aligned.
 * sq_err  : out, device, one int64 per tile (row-major tile order): the
 *           tile's summed squared error in grid units^2; may be NULL.
 * scratch : device, at least tfx_exl3_encode_scratch_bytes(...) bytes (per
 *           concurrent tile: two 2^16 int32 cost arrays and 256 x 2^(16-bits)
 *           argmin bytes); 16-byte aligned; caller-owned.
 * max_ctas: tiles encoded at once (0: one per SM); the scratch size depends on it.
 * K, N multiples of 16, bits 1..8. Enqueued on `stream`; the words equal the
 * CPU oracle's bit for bit (all decisions are integer). */
int tfx_exl3_encode_scratch_bytes(int K, int N, int bits, int max_ctas, size_t* bytes);
int tfx_exl3_encode(const int16_t* targets, int K, int N, int bits, uint32_t* trellis, int64_t* sq_err, void* scratch,
                    size_t scratch_bytes, int max_ctas, cudaStream_t stream);

/* Measurement hook: the next linear/group call on this thread records
 * `before` just before its linear-kernel launch and `after` just after it,
 * on the call's stream, then forgets both. Either may be NULL. Inside a
 * stream capture the records become external event-record nodes, so the
 * events can be timed when the graph is replayed. */
int tfx_exl3_debug_mark_events(cudaEvent_t before, cudaEvent_t after);

const char* tfx_exl3_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TFX_EXL3_H */
