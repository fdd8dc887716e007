// Host-side helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/flce.h"

namespace flce {

// Number of SMs of the current device (cached per device id).
int sm_count();

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t dtype_size(int dt) { return dt == FLCE_BF16 ? 2 : 4; }

inline bool valid_dtype(int dt) { return dt == FLCE_BF16 || dt == FLCE_F32; }

inline bool valid_reduction(int r) { return r == FLCE_SUM || r == FLCE_MEAN; }

// Records a failed CUDA call for flce_last_cuda_error (per thread).
void record_cuda_error(cudaError_t e, const char* where);

// Maps a CUDA result to a status, recording failures.
inline int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return FLCE_OK;
  record_cuda_error(e, where);
  return FLCE_ECUDA;
}

// Launch-time error of the last kernel launch (configuration errors only).
inline int launch_status(const char* where = "kernel launch") {
  return cuda_status(cudaGetLastError(), where);
}

// Per-row loss reduction shared by both operations: sums loss_rows[0..N) in a
// fixed order in fp64, counts valid labels exactly, applies the reduction.
int launch_finalize(const float* loss_rows, const int64_t* labels, int64_t N, int64_t V,
                    int64_t ignore_index, int reduction, int64_t num_label_tokens, float* loss,
                    int64_t* n_valid, cudaStream_t stream);

}  // namespace flce
