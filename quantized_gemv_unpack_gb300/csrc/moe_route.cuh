// Top-k routing of the MoE decode ("Nemotron 3.5 Bolt", expert top-K routing),
// run in shared memory by every CTA of the expert kernels (moe.cu and the
// byte-lookup experts of lut.cu): the same inputs give every CTA the same
// result, so no launch is spent on it and no CTA waits for another.
//
// Each (token, expert) logit becomes a 64-bit key, its order-preserving bits
// (NaN as -inf, -0 as +0) above the complement of the expert index, so that the
// keys of a token are distinct and ordered as the selection wants: larger logit
// first, equal logits lower expert first. One warp per token holds the token's
// keys in registers (expert lane + 32 i in slot i), each lane sorts its own
// keys, and k rounds of a warp maximum over the lanes' largest remaining keys
// take the selection out in rank order (the winning lane drops its largest).
// The softmax over the k selected logits is fp32: each selected entry's thread
// sums the k exponentials in rank order and divides its own. Then one thread per
// (token, expert) pair counts the pairs before it in expert, then token order
// (its position) and the pairs of its expert; the first pair of each expert
// heads a slot, numbered by the heads of smaller experts.
#pragma once

#include "qmv_internal.cuh"

namespace qmv {

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
  int pair_token[kMaxPairs], pair_expert[kMaxPairs];
  float pair_prob[kMaxPairs];
  int exp[kMaxTokens][kMaxTopk];
  float prob[kMaxTokens][kMaxTopk];
  int head_expert[kMaxPairs];  // the expert of a slot-heading pair (by pair index), else -1
};

__device__ __forceinline__ unsigned long long route_key(float v, int e) {
  if (v != v) v = -INFINITY;
  v += 0.f;  // -0 -> +0
  const uint32_t b = __float_as_uint(v);
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 8) | (uint32_t)(255 - e);
}
__device__ __forceinline__ float route_key_value(unsigned long long k) {
  const uint32_t o = (uint32_t)(k >> 8);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ void cas_desc(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Warp `t`'s top-k of token t's logits into R.exp[t] / R.prob[t] (rank order);
// KPL keys per lane (E <= 32 KPL).
template <int KPL>
__device__ __forceinline__ void route_topk_warp(const MoeRouting& a, MoeRoute& R, int t) {
  const int lane = threadIdx.x & 31;
  unsigned long long k[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    k[i] = e < a.E ? route_key(a.logits[(size_t)t * a.E + e], e) : 0ull;  // 0: below every key
  }
  // sort the lane's keys, largest first (odd-even transposition: KPL rounds)
#pragma unroll
  for (int r = 0; r < KPL; ++r)
#pragma unroll
    for (int i = r & 1; i + 1 < KPL; i += 2) cas_desc(k[i], k[i + 1]);
  for (int r = 0; r < a.topk; ++r) {
    unsigned long long best = k[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long v = __shfl_xor_sync(0xffffffffu, best, o);
      best = v > best ? v : best;
    }
    if (k[0] == best) {  // keys are distinct: one lane drops its largest
#pragma unroll
      for (int i = 0; i + 1 < KPL; ++i) k[i] = k[i + 1];
      k[KPL - 1] = 0ull;
    }
    if (lane == 0) {
      R.exp[t][r] = 255 - (int)(best & 0xFFu);
      R.prob[t][r] = route_key_value(best);
    }
  }
}

// Called by all threads of the CTA (blockDim.x a multiple of 32, at least 32 M and
// 64); E <= 256, k <= 8, M <= 8. Ends with a CTA barrier.
__device__ inline void route(const MoeRouting& a, MoeRoute& R) {
  const int warp = threadIdx.x >> 5;
  if (warp < a.M) {
    if (a.E <= 128) route_topk_warp<4>(a, R, warp);
    else route_topk_warp<8>(a, R, warp);
  }
  __syncthreads();
  // softmax over each token's k selected logits: every thread of the token's k
  // takes the sum of the exponentials in rank order and divides its own
  const int st = threadIdx.x / kMaxTopk, sr = threadIdx.x % kMaxTopk;
  float ex = 0.f;
  if (st < a.M && sr < a.topk) {
    const float mx = R.prob[st][0];
    float z = 0.f;
    for (int r = 0; r < a.topk; ++r) z += expf(R.prob[st][r] - mx);
    ex = expf(R.prob[st][sr] - mx) / z;
  }
  __syncthreads();
  if (st < a.M && sr < a.topk) R.prob[st][sr] = ex;
  __syncthreads();
  // pairs ordered by expert, then token (a token's k experts are distinct)
  const int P = a.M * a.topk;
  const int pi = threadIdx.x;
  int pos = 0, cnt = 0, before = 0, pe = 0, pt = 0;
  if (pi < P) {
    pt = pi / a.topk;
    pe = R.exp[pt][pi - pt * a.topk];
    for (int tj = 0; tj < a.M; ++tj)
      for (int rj = 0; rj < a.topk; ++rj) {
        const int ej = R.exp[tj][rj];
        pos += ej < pe || (ej == pe && tj < pt);
        cnt += ej == pe;
        before += ej == pe && tj < pt;
      }
    R.pair_token[pos] = pt;
    R.pair_expert[pos] = pe;
    R.pair_prob[pos] = R.prob[pt][pi - pt * a.topk];
    R.head_expert[pi] = before == 0 ? pe : -1;
  }
  __syncthreads();
  if (pi < P && before == 0) {
    int slot = 0;
    for (int j = 0; j < P; ++j) {
      const int hj = R.head_expert[j];
      slot += hj >= 0 && hj < pe;
    }
    R.slot_expert[slot] = pe;
    R.slot_first[slot] = pos;
    R.slot_count[slot] = cnt;
  }
  if (threadIdx.x == 0) {
    int ns = 0;
    for (int j = 0; j < P; ++j) ns += R.head_expert[j] >= 0;
    R.n_slots = ns;
  }
  __syncthreads();
}

}  // namespace qmv
