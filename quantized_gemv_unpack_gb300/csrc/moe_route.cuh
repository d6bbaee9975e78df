// Top-k routing of the MoE decode ("Nemotron 3.5 Bolt", expert top-K routing),
// run in shared memory by every CTA of the expert kernels (moe.cu and the
// byte-lookup experts of lut.cu): the same inputs give every CTA the same
// result, so no launch is spent on it and no CTA waits for another.
//
// One warp per token takes the top-k of its E logits (equal logits: lower
// expert first) by k rounds of a warp arg-max, and the softmax over the k
// selected logits in fp32; then one thread per expert counts its (token,
// expert) pairs and a block scan orders the pairs by expert and token and lists
// each active expert once (a slot).
#pragma once

#include "qmv_internal.cuh"

namespace qmv {

constexpr int kMaxMoeWarps = 20;
constexpr int kMaxTopk = 8;
constexpr int kMaxTokens = 8;
constexpr int kMaxExperts = 256;
constexpr int kMaxPairs = kMaxTokens * kMaxTopk;

// The routing inputs.
struct MoeRouting {
  const float* logits;  // [M][E]
  int E, topk, M;
};

// Routing of the M tokens, in shared memory.
struct MoeRoute {
  int n_slots;
  int slot_expert[kMaxPairs], slot_first[kMaxPairs], slot_count[kMaxPairs];
  int pair_token[kMaxPairs];
  float pair_prob[kMaxPairs];
  int exp[kMaxTokens][kMaxTopk];
  float prob[kMaxTokens][kMaxTopk];
  int wp[kMaxMoeWarps], ws[kMaxMoeWarps];
};

// Called by all threads of the CTA (blockDim.x >= E); ends with a CTA barrier.
__device__ inline void route(const MoeRouting& a, MoeRoute& R) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < a.M) {
    // the lane's logits in registers and a bit mask of the entries taken (or past
    // E), so that nothing is indexed at run time
    const float* lg = a.logits + (size_t)warp * a.E;
    float v[kMaxExperts / 32];
    uint32_t taken = 0u;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = i * 32 + lane;
      v[i] = e < a.E ? lg[e] : -INFINITY;
      if (e >= a.E) taken |= 1u << i;
    }
    for (int r = 0; r < a.topk; ++r) {
      // best remaining (value, index) of this lane, then across the warp; equal
      // values keep the lower index
      float bv = -INFINITY;
      int bi = 1 << 30;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i)
        if (!((taken >> i) & 1u) && (bi == (1 << 30) || v[i] > bv)) bv = v[i], bi = i * 32 + lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) bv = ov, bi = oi;
      }
      if (bi < a.E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == 0) {
        R.exp[warp][r] = bi < a.E ? bi : 0;
        R.prob[warp][r] = bv;
      }
    }
    __syncwarp();
    if (lane == 0) {
      const float mx = R.prob[warp][0];
      float z = 0.f;
      for (int r = 0; r < a.topk; ++r) {
        R.prob[warp][r] = expf(R.prob[warp][r] - mx);
        z += R.prob[warp][r];
      }
      for (int r = 0; r < a.topk; ++r) R.prob[warp][r] /= z;
    }
  }
  __syncthreads();
  // pairs ordered by expert, then token: thread e counts expert e's pairs, a
  // block-wide exclusive scan of (pairs, active) gives its first pair and its
  // slot, and it writes its pairs in token order
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < a.E)
    for (int t = 0; t < a.M; ++t)
      for (int r = 0; r < a.topk; ++r) cnt += R.exp[t][r] == e;
  const int act = cnt > 0;
  int pc = cnt, sc = act;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int up = __shfl_up_sync(0xffffffffu, pc, o), us = __shfl_up_sync(0xffffffffu, sc, o);
    if (lane >= o) {
      pc += up;
      sc += us;
    }
  }
  if (lane == 31) {
    R.wp[warp] = pc;
    R.ws[warp] = sc;
  }
  __syncthreads();
  int base_p = 0, base_s = 0;
  for (int w = 0; w < warp; ++w) {
    base_p += R.wp[w];
    base_s += R.ws[w];
  }
  if (act) {
    int np = base_p + pc - cnt;
    const int slot = base_s + sc - 1;
    R.slot_expert[slot] = e;
    R.slot_first[slot] = np;
    R.slot_count[slot] = cnt;
    for (int t = 0; t < a.M; ++t)
      for (int r = 0; r < a.topk; ++r)
        if (R.exp[t][r] == e) {
          R.pair_token[np] = t;
          R.pair_prob[np] = R.prob[t][r];
          ++np;
        }
  }
  if (threadIdx.x == blockDim.x - 1) R.n_slots = base_s + sc;
  __syncthreads();
}

}  // namespace qmv
