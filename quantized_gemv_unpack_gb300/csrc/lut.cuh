// Byte-lookup ternary matvec (lut.cu): the entry points' host side.
#pragma once

#include "qmv_internal.cuh"

namespace qmv {

// Check a QMV_TERNARY2_LUT descriptor (format, shape and section layout).
int check_lut_desc(const qmv_desc* d);
// n matvecs at M = 1 in one launch; the tasks' descriptors are checked here.
int run_lut(const qmv_task* tasks, int n, cudaStream_t s);

}  // namespace qmv
