// Internal declarations shared by the translation units of libqmv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmv.h"

namespace qmv {

// ----------------------------------------------------------------------------- host helpers

// Record a message for qmv_last_error() and return `status`.
int fail(int status, const char* fmt, ...);
// Record a CUDA failure (with the CUDA error string) and return QMV_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* what);
// Device address of the current device's error word (set up once per device).
int* device_error_word();
// Multiprocessor count of the current device.
int sm_count();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_desc(const qmv_desc* d, int format);
// Raise the kernel's dynamic shared memory limit when needed and return how
// many CTAs of `threads` threads fit on one SM (cached per kernel and size).
int kernel_fit(const void* kernel, int threads, size_t smem, int* per_sm);

// ----------------------------------------------------------------------------- matvec batch

constexpr int kThreads = 256;      // 8 warps per CTA
constexpr int kMaxTasks = QMV_MAX_BATCH;

// One matvec of a persistent launch. Tiles of gemv_rows_per_tile(M) rows are
// numbered across tasks: task i owns tiles [tile0, tile0 + ceil(N / rows)).
struct GemvTask {
  const uint32_t* codes;   // section 0
  const uint16_t* scales;  // section 1 (fp16 bits)
  const uint16_t* x;       // bf16 bits [M][ldx]
  float* y;                // [M][ldy]
  int32_t N, K;
  int32_t ldx, ldy;
  int32_t tile0;
  int32_t pad;
};

struct GemvBatch {
  int32_t n_tasks;
  int32_t n_tiles;
  int32_t kc;              // activation chunk staged in shared memory (elements)
  int32_t pad;
  GemvTask t[kMaxTasks];
};

// Rows per tile of the persistent matvec kernel for M activation rows.
int gemv_rows_per_tile(int M);
// Launch the persistent matvec kernel for `format` (QMV_TERNARY2 / QMV_INT4);
// sets b.kc. M in 1..8.
int launch_gemv(int format, GemvBatch& b, int M, int max_K, cudaStream_t s);

}  // namespace qmv
