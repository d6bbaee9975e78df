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

// Ternary/INT4 scale section: fp16 scales in the record order of the codes, one
// record of 16 rows x 8 blocks (256 bytes) per (16-row group, 1024-column step),
// rows past N and blocks past K/128 zero. scale_steps(K) steps per row.
__host__ __device__ __forceinline__ int64_t scale_steps(int64_t K) { return (K / 128 + 7) / 8; }
__host__ __device__ __forceinline__ int64_t scale_index(int64_t n, int64_t b, int64_t steps) {
  return ((n / 16) * steps + b / 8) * 128 + (n % 16) * 8 + b % 8;
}

int check_desc(const qmv_desc* d, int format);
// Raise the kernel's dynamic shared memory limit when needed and return how
// many CTAs of `threads` threads fit on one SM (cached per kernel and size).
int kernel_fit(const void* kernel, int threads, size_t smem, int* per_sm);

// ----------------------------------------------------------------------------- matvec batch

constexpr int kConsumerWarps = 16;                      // decode warps per CTA (4 per SM sub-partition)
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kMaxTasks = QMV_MAX_BATCH;
constexpr int kMaxCtas = 256;                           // persistent grid: at most one CTA per SM

// One matvec of a persistent launch. Tiles of rows_per_tile rows are numbered
// across tasks: task i owns tiles [tile0, tile0 + ceil(N / rows_per_tile)).
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
  int32_t rows_per_tile;
  int32_t n_ctas;
  // testing only (QMV_FLAG_TEST_WAIT_TIMEOUT): > 0 makes the kernel's first
  // wait one that nothing completes, limited to this many microseconds
  uint32_t test_wait_us;
  // CTA c processes the contiguous tile range [cta_tile[c], cta_tile[c+1]),
  // cut so every CTA streams about the same number of bytes
  int32_t cta_tile[kMaxCtas + 1];
  // decode constants, passed at run time so they live in registers: {mask,
  // base} make each decode a single three-input logic op, and the shift
  // multipliers/amounts pin each shift to the integer-multiply or the
  // shift unit (see gemv.cu)
  uint32_t magic[10];
  int* err;                // device error word (timeouts of bounded waits)
  GemvTask t[kMaxTasks];
};

// Launch the persistent fp16-FMA matvec kernel for `format` (QMV_TERNARY2 /
// QMV_INT4) over b.t[0 .. b.n_tasks); fills the tiling fields of b. M in 1..8.
int launch_gemv(int format, GemvBatch& b, int M, cudaStream_t s);
// The tensor-core matvec kernel (gemv_mma.cu), same contract, M in 1..16.
int launch_gemv_mma(int format, GemvBatch& b, int M, cudaStream_t s);
// Flagged sparse ternary (sparse.cu): descriptor check, and n matvecs with M
// activation rows in one launch (descriptors already checked).
int check_sparse_desc(const qmv_desc* d);
int run_sparse(const qmv_desc* const* descs, const void* const* ws, const void* const* xs, const int64_t* ldx,
               float* const* ys, const int64_t* ldy, int n, int M, cudaStream_t s);

// From this many activation rows on, the entry points use the tensor-core
// kernel (unless qmv_desc.flags forces one of the two): the fp16-FMA kernel's
// cost grows with M; measured on the INT4 layer set, the 4096 x 4096 ternary
// matrix and the ternary stack it is ahead only for ternary at M = 1 (INT4
// decodes more words per weight byte, so the tensor-core kernel wins there from
// M = 1).
inline int mma_min_m(int format) { return format == QMV_INT4 ? 1 : 2; }

}  // namespace qmv
