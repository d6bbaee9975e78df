// Byte-lookup ternary matvec (lut.cu): the entry points' host side.
#pragma once

#include "qmv_internal.cuh"

namespace qmv {

// Check a QMV_TERNARY2_LUT descriptor (format, shape and section layout).
int check_lut_desc(const qmv_desc* d);
// n matvecs at M = 1 in one launch; the tasks' descriptors are checked here.
int run_lut(const qmv_task* tasks, int n, cudaStream_t s);

// The MoE decode over experts in the lookup layout (arguments already checked
// by moe_qmv_run): one (token, expert) pair per task, routing in every CTA,
// workspace offsets as moe_qmv_run's layout; a gate|up and a down launch.
struct LutMoeCall {
  const unsigned char* gu_codes;  // expert 0's [gate; up] codes (2I x H); expert e at + e * stride
  const unsigned char* dn_codes;  // expert 0's down codes (H x I)
  int64_t stride;
  const float* logits;
  int E, topk, M;
  int64_t H, I;
  const uint16_t* x;
  int64_t ldx;
  float* y;
  int64_t ldy;
  unsigned char* ws;
  int64_t off_slot_expert, off_slot_first, off_slot_count, off_pair_token, off_pair_prob, off_gu;
};
int run_lut_moe(const LutMoeCall& c, cudaStream_t s);

}  // namespace qmv
