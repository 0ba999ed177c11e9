// Internal interface between the C-ABI translation units (not installed).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>

#include "../../include/tfx_exl3.h"
#include "exl3_kernels.cuh"

namespace tfx {

// Scratch of one call, per member: rotated x (fragment order), subtree slabs, counters.
struct Scratch {
  uint2* xf[3];
  float* partial[3];
  int* counters[3];
  int* err;    // device error word (a bounded wait gave up)
  float* lev;  // tensor-core chunk-tree level slots (null: passes of at most 64 rows above 128 rows)
};

// The counter buffer of a weight starts with this many ints: word 0 is the
// device error word, the rest pad the counters to 16 bytes.
constexpr int kErrorInts = 4;

// K chunks of the summation order: a pure function of K.
int chunks_of(int K);
// Bytes of rotated x, slabs and counters one weight needs for up to `rows` rows.
size_t xf_bytes_needed(const tfx_exl3_weight* w, int rows);
size_t partial_bytes_needed(const tfx_exl3_weight* w, int rows);
size_t counter_bytes_needed(const tfx_exl3_weight* w, int rows);
size_t level_bytes_needed(int rows);
// Enqueue the rotation and the linear launch for validated members on `s`;
// ldy / col0 give each member's output window (null: N and 0).
int launch_layer(tfx_exl3_weight* const ws[], int count, const void* x, int rows, void* const ys[],
                 const int64_t* ldy, const int* col0, cudaStream_t s, const Scratch& sc, int pdl);
int report_error(int code, const char* msg);

}  // namespace tfx
