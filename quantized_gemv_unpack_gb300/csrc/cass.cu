// Cassandra lossless bf16 split ("Cassandra", sections 3.1-3.3): the host-side
// offline transform and the GPU draft / target paths.
//
// Offline (host): Wanda value pruning keeps the K/2 largest |w| * ||X[:,j]||_2
// of every row (bitmap), kept values keep sign + 3 high mantissa bits in the
// speculation data and 4 low mantissa bits in the verification data, their
// exponents are ranked by frequency over the whole tensor and written as unary
// codes (rank r = r zeros then a one), pruned values go to the verification
// data as raw bf16.
//
// GPU: one warp per row, rows strided over a persistent grid. Phase A decodes
// the row's unary exponent stream: each lane takes one 32-bit word, counts the
// codewords ending in it (__popc), an inclusive warp scan turns the counts into
// codeword indices, and an exclusive warp max-scan of each word's last one bit
// (carried across 32-word chunks) gives every codeword's start, so a lane can
// turn each set bit into a rank = zeros since the previous one and look the
// exponent up in the codebook. Exponents land in shared memory in kept-value
// order. Phase B walks the bitmap 32 columns at a time: lane l owns column
// 32*i + l, its kept index is the number of kept columns before it
// (__popc(word & lanemask_lt) plus the running count), its pruned index is
// column - kept index. The draft value is S<<15 | E<<7 | m_hi<<4 (pruned: +0),
// the target value adds m_lo (pruned: the raw verification bits); either is
// widened to fp32 (exact) and multiplied into fp32 accumulators per activation
// row. Every loop is bounded by the row's sizes; inconsistent streams set
// QMV_ERR_CORRUPT in the device error word.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "qmv_internal.cuh"

namespace qmv {
namespace {

constexpr int kCassWarpsMax = 16;

struct CassArgs {
  const uint32_t* bitmap;    // [N][K/32]
  const uint32_t* signmant;  // [N][K/16]
  const uint32_t* stream;    // unary words
  const uint32_t* rowstart;  // [N+1]
  const uint8_t* codebook;   // [256]
  const uint16_t* pruned;    // [N][K/2]
  const uint32_t* mlo;       // [N][K/16]
  const uint16_t* x;         // bf16 [M][ldx]
  float* y;                  // [M][ldy] or null
  uint16_t* w_out;           // [N][K] or null
  int64_t stream_words;
  int N, K, ldx, ldy, n_symbols;
  int* err;
};

__device__ __forceinline__ void flag(int* err) { atomicCAS(err, 0, (int)QMV_ERR_CORRUPT); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <int MT, bool TARGET>
__global__ void __launch_bounds__(kCassWarpsMax * 32) cass_kernel(const CassArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int K = a.K;
  const int K2 = K / 2;
  const int nwarps = blockDim.x / 32;
  float* xs = reinterpret_cast<float*>(smem);                       // [MT][K] fp32
  uint8_t* cb = smem + (size_t)MT * K * 4;                           // [256]
  // per-warp buffers: bitmap[K/32] words, signmant[K/16] words, (target: mlo[K/16] words,
  // pruned[K/2] halves), exps[K/2] bytes
  const size_t per_warp = ((size_t)K2 + (size_t)K / 8 + (size_t)K / 4 + (TARGET ? (size_t)K / 4 + (size_t)K : 0) + 15) / 16 * 16;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* wb = smem + (size_t)MT * K * 4 + 256 + (size_t)warp * per_warp;
  uint32_t* bm_s = reinterpret_cast<uint32_t*>(wb);
  uint32_t* sm_s = bm_s + K / 32;
  uint32_t* lo_s = sm_s + K / 16;
  uint16_t* pr_s = reinterpret_cast<uint16_t*>(lo_s + (TARGET ? K / 16 : 0));
  uint8_t* exps = reinterpret_cast<uint8_t*>(pr_s + (TARGET ? K2 : 0));

  for (int i = threadIdx.x; i < 256; i += blockDim.x) cb[i] = a.codebook[i];
  for (int m = 0; m < MT; ++m)
    for (int j = threadIdx.x; j < K; j += blockDim.x)
      xs[(size_t)m * K + j] = __uint_as_float((uint32_t)a.x[(size_t)m * a.ldx + j] << 16);
  __syncthreads();

  const uint32_t below = lanemask_lt();
  const int gw = blockIdx.x * nwarps + warp;
  const int stride = gridDim.x * nwarps;
  for (int n = gw; n < a.N; n += stride) {
    // ---- stage the row's fixed-size sections (all loads in flight together);
    // rows are 16-byte aligned in global memory when K is a multiple of 128
    if (K % 128 == 0) {
      const uint4* bm = reinterpret_cast<const uint4*>(a.bitmap + (size_t)n * (K / 32));
      const uint4* sm = reinterpret_cast<const uint4*>(a.signmant + (size_t)n * (K / 16));
      for (int i = lane; i < K / 128; i += 32) reinterpret_cast<uint4*>(bm_s)[i] = __ldg(bm + i);
      for (int i = lane; i < K / 64; i += 32) reinterpret_cast<uint4*>(sm_s)[i] = __ldg(sm + i);
      if (TARGET) {
        const uint4* lo = reinterpret_cast<const uint4*>(a.mlo + (size_t)n * (K / 16));
        const uint4* pr = reinterpret_cast<const uint4*>(a.pruned + (size_t)n * K2);
        for (int i = lane; i < K / 64; i += 32) reinterpret_cast<uint4*>(lo_s)[i] = __ldg(lo + i);
        for (int i = lane; i < K / 16; i += 32) reinterpret_cast<uint4*>(pr_s)[i] = __ldg(pr + i);
      }
    } else {
      const uint32_t* bm = a.bitmap + (size_t)n * (K / 32);
      const uint32_t* sm = a.signmant + (size_t)n * (K / 16);
      for (int i = lane; i < K / 32; i += 32) bm_s[i] = __ldg(bm + i);
      for (int i = lane; i < K / 16; i += 32) sm_s[i] = __ldg(sm + i);
      if (TARGET) {
        const uint32_t* lo = a.mlo + (size_t)n * (K / 16);
        const uint16_t* pr = a.pruned + (size_t)n * K2;
        for (int i = lane; i < K / 16; i += 32) lo_s[i] = __ldg(lo + i);
        for (int i = lane; i < K2; i += 32) pr_s[i] = __ldg(pr + i);
      }
    }

    // ---- phase A: unary exponent codes -> exps[kept index]
    uint32_t s0 = __ldg(a.rowstart + n), s1 = __ldg(a.rowstart + n + 1);
    if (s1 < s0 || (int64_t)s1 > a.stream_words) {
      if (lane == 0) flag(a.err);
      s1 = s0;
    }
    const int nwords = (int)(s1 - s0);
    int count = 0;       // codewords so far (warp-uniform)
    int carry = -1;      // row-relative bit position of the last one so far
    for (int c = 0; c < nwords; c += 32) {
      const int wi = c + lane;
      const uint32_t w = wi < nwords ? __ldg(a.stream + s0 + wi) : 0u;
      const int cnt = __popc(w);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int lastpos = w ? wi * 32 + 31 - __clz(w) : -1;
      int mx = lastpos;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, mx, o);
        if (lane >= o) mx = max(mx, t);
      }
      int prev = __shfl_up_sync(0xffffffffu, mx, 1);
      prev = lane == 0 ? carry : max(prev, carry);
      int k = count + incl - cnt;
      uint32_t bits = w;
      bool bad = false;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        const int pos = wi * 32 + b;
        const int rank = pos - prev - 1;
        prev = pos;
        uint8_t e = 0;
        if (rank < a.n_symbols) e = cb[rank]; else bad = true;
        if (k < K2) exps[k] = e; else bad = true;
        ++k;
      }
      if (bad) flag(a.err);
      count += __shfl_sync(0xffffffffu, incl, 31);
      carry = max(carry, __shfl_sync(0xffffffffu, mx, 31));
    }
    if (count != K2 && lane == 0) flag(a.err);
    __syncwarp();

    // ---- phase B: rebuild each column's bf16 value and accumulate w * x,
    // four bitmap words per iteration (their kept counts prefix-summed first)
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    int kbase = 0;
    uint16_t* wrow = a.w_out ? a.w_out + (size_t)n * K : nullptr;
    auto column = [&](uint32_t word, int it, int kb) {
      const int j = it * 32 + lane;
      const bool kept = (word >> lane) & 1u;
      const int kidx = kb + __popc(word & below);
      uint32_t v = 0;
      if (kept) {
        if (kidx < K2) {
          const uint32_t nib = (sm_s[kidx >> 3] >> ((kidx & 7) * 4)) & 0xFu;
          v = ((nib >> 3) << 15) | ((uint32_t)exps[kidx] << 7) | ((nib & 7u) << 4);
          if (TARGET) v |= (lo_s[kidx >> 3] >> ((kidx & 7) * 4)) & 0xFu;
        }
      } else if (TARGET) {
        const int pidx = j - kidx;
        if (pidx < K2) v = pr_s[pidx];
      }
      if (wrow) wrow[j] = (uint16_t)v;
      const float wf = __uint_as_float(v << 16);
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(wf, xs[(size_t)m * K + j], acc[m]);
    };
    int it = 0;
    for (; it + 4 <= K / 32; it += 4) {
      const uint4 w4 = reinterpret_cast<const uint4*>(bm_s)[it >> 2];
      const int k1 = kbase + __popc(w4.x), k2 = k1 + __popc(w4.y), k3 = k2 + __popc(w4.z);
      column(w4.x, it, kbase);
      column(w4.y, it + 1, k1);
      column(w4.z, it + 2, k2);
      column(w4.w, it + 3, k3);
      kbase = k3 + __popc(w4.w);
    }
    for (; it < K / 32; ++it) {
      const uint32_t word = bm_s[it];
      column(word, it, kbase);
      kbase += __popc(word);
    }
    if (kbase != K2 && lane == 0) flag(a.err);
    if (a.y) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = acc[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) a.y[(size_t)m * a.ldy + n] = v;
      }
    }
    __syncwarp();  // the staged row buffers are reused by the next row
  }
}

// ----------------------------------------------------------------------------- Cassandra-2 (MX)

struct CassMxArgs {
  const uint32_t* bitmap;    // [N][K/32]
  const uint8_t* gexp;       // [N][K/64]
  const uint32_t* signs;     // [N][K/64]
  const uint32_t* dnib;      // [N][K/16]
  const uint32_t* lnib;      // [N][K/16]
  const uint16_t* pruned;    // [N][K/2]
  const uint16_t* x;         // bf16 [M][ldx]
  float* y;                  // [M][ldy] or null
  uint16_t* w_out;           // [N][K] or null
  int N, K, ldx, ldy;
  int* err;
};

__host__ __device__ inline size_t cassmx_per_warp(size_t K, bool target) {
  // bitmap, signs, dnib, group scales (+ target: lnib, pruned)
  return (K / 8 + K / 16 + K / 4 + K / 16 + (target ? K / 4 + K : 0) + 15) / 16 * 16;
}

// One warp per row, rows strided over a persistent grid. The row's sections are
// staged in shared memory together with one fp32 scale per group of 32 kept
// values (2^(g - 134) for the target, 2^(g - 130) for the draft), so a kept
// column's value is one nibble lookup times its group's scale: no per-value
// exponent decode. Lane l owns column 32*i + l of each bitmap word, as in the
// Cassandra-1 kernel; values are exact in fp32 and in bf16.
template <int MT, bool TARGET>
__global__ void __launch_bounds__(kCassWarpsMax * 32) cassmx_kernel(const CassMxArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int K = a.K;
  const int K2 = K / 2;
  const int KG = K / 64;
  const int nwarps = blockDim.x / 32;
  float* xs = reinterpret_cast<float*>(smem);  // [MT][K] fp32
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* wb = smem + (size_t)MT * K * 4 + (size_t)warp * cassmx_per_warp(K, TARGET);
  uint32_t* bm_s = reinterpret_cast<uint32_t*>(wb);
  uint32_t* sg_s = bm_s + K / 32;
  uint32_t* dn_s = sg_s + K / 64;
  float* sc_s = reinterpret_cast<float*>(dn_s + K / 16);
  uint32_t* ln_s = reinterpret_cast<uint32_t*>(sc_s + KG);
  uint16_t* pr_s = reinterpret_cast<uint16_t*>(ln_s + (TARGET ? K / 16 : 0));

  for (int m = 0; m < MT; ++m)
    for (int j = threadIdx.x; j < K; j += blockDim.x)
      xs[(size_t)m * K + j] = __uint_as_float((uint32_t)a.x[(size_t)m * a.ldx + j] << 16);
  __syncthreads();

  const uint32_t below = lanemask_lt();
  const int gw = blockIdx.x * nwarps + warp;
  const int stride = gridDim.x * nwarps;
  for (int n = gw; n < a.N; n += stride) {
    for (int i = lane; i < K / 32; i += 32) bm_s[i] = __ldg(a.bitmap + (size_t)n * (K / 32) + i);
    for (int i = lane; i < K / 64; i += 32) sg_s[i] = __ldg(a.signs + (size_t)n * (K / 64) + i);
    for (int i = lane; i < K / 16; i += 32) dn_s[i] = __ldg(a.dnib + (size_t)n * (K / 16) + i);
    for (int i = lane; i < KG; i += 32)
      sc_s[i] = ldexpf(1.f, (int)__ldg(a.gexp + (size_t)n * KG + i) - (TARGET ? 134 : 130));
    if (TARGET) {
      for (int i = lane; i < K / 16; i += 32) ln_s[i] = __ldg(a.lnib + (size_t)n * (K / 16) + i);
      for (int i = lane; i < K2; i += 32) pr_s[i] = __ldg(a.pruned + (size_t)n * K2 + i);
    }
    __syncwarp();

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    uint16_t* wrow = a.w_out ? a.w_out + (size_t)n * K : nullptr;
    int kbase = 0;
    bool bad = false;
    for (int it = 0; it < K / 32; ++it) {
      const uint32_t word = bm_s[it];
      const int j = it * 32 + lane;
      const int kidx = kbase + __popc(word & below);
      float v = 0.f;
      if ((word >> lane) & 1u) {
        if (kidx < K2) {
          const uint32_t sh = (kidx & 7) * 4;
          uint32_t mag = (dn_s[kidx >> 3] >> sh) & 0xFu;
          if (TARGET) mag = (mag << 4) | ((ln_s[kidx >> 3] >> sh) & 0xFu);
          v = (float)mag * sc_s[kidx >> 5];
          if ((sg_s[kidx >> 5] >> (kidx & 31)) & 1u) v = -v;
        } else {
          bad = true;
        }
      } else if (TARGET) {
        const int pidx = j - kidx;
        if (pidx < K2) v = __uint_as_float((uint32_t)pr_s[pidx] << 16);
        else bad = true;
      }
      if (wrow) wrow[j] = (uint16_t)(__float_as_uint(v) >> 16);
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(v, xs[(size_t)m * K + j], acc[m]);
      kbase += __popc(word);
    }
    if (bad || (kbase != K2 && lane == 0)) flag(a.err);
    if (a.y) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float t = acc[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) a.y[(size_t)m * a.ldy + n] = t;
      }
    }
    __syncwarp();  // the staged row buffers are reused by the next row
  }
}

template <bool TARGET>
int launch_cassmx(const CassMxArgs& a, int M, cudaStream_t s) {
  const size_t K = a.K;
  const size_t per_warp = cassmx_per_warp(K, TARGET);
  const size_t fixed = (size_t)M * K * 4;
  const size_t cap = 227 * 1024 - 1024;
  if (fixed + per_warp > cap) return fail(QMV_ERR_UNSUPPORTED, "K=%zu with M=%d does not fit shared memory", K, M);
  const int warps = (int)std::min<size_t>(kCassWarpsMax, (cap - fixed) / per_warp);
  const size_t smem = fixed + per_warp * warps;
  const void* kern = nullptr;
  switch (M) {
#define QMV_CASSMX_CASE(m) \
  case m: kern = (const void*)cassmx_kernel<m, TARGET>; break;
    QMV_CASSMX_CASE(1) QMV_CASSMX_CASE(2) QMV_CASSMX_CASE(3) QMV_CASSMX_CASE(4)
    QMV_CASSMX_CASE(5) QMV_CASSMX_CASE(6) QMV_CASSMX_CASE(7) QMV_CASSMX_CASE(8)
#undef QMV_CASSMX_CASE
    default: return fail(QMV_ERR_ARG, "M=%d outside 1..8", M);
  }
  int per_sm = 0;
  int rc = kernel_fit(kern, warps * 32, smem, &per_sm);
  if (rc) return rc;
  const int grid = std::max(1, std::min(sm_count() * per_sm, (a.N + warps - 1) / warps));
  void* args[] = {const_cast<CassMxArgs*>(&a)};
  cudaError_t e = cudaLaunchKernel(kern, grid, warps * 32, args, smem, s);
  if (e != cudaSuccess) return cuda_fail(e, "cassandra-2 launch");
  return QMV_OK;
}

// ----------------------------------------------------------------------------- online KV encoder

struct KvEncArgs {
  const uint16_t* v;         // bf16 [T][ld]
  int64_t ld;
  int T, D, slot_words;
  uint32_t* bitmap;          // the Cassandra-1 sections of the output buffer
  uint32_t* signmant;
  uint32_t* stream;
  uint32_t* rowstart;
  uint8_t* codebook;
  uint16_t* pruned;
  uint32_t* mlo;
  unsigned char* base;       // the output buffer, for its section gaps
  int64_t gap_begin[7], gap_end[7];
  uint32_t cb_words[64];     // codebook bytes in rank order
  int* err;
};

constexpr int kEncWarps = 4;

__device__ __forceinline__ uint32_t magnitude_key(uint32_t b) {
  // |v| ordering of bf16 bits; Inf and NaN both as +inf
  return ((b >> 7) & 0xFFu) == 0xFFu ? 0x7F80u : (b & 0x7FFFu);
}

// Among the 256 bins of hist (one digit of the key), the digit d at which the
// count of keys with digit > d stays below `need` and with digit >= d reaches
// it; returns d and sets *above to the count with digit > d. Warp-collective.
__device__ int select_digit(const int* hist, int need, int* above) {
  const int lane = threadIdx.x & 31;
  // lane l holds bins 255 - 8l .. 248 - 8l (descending)
  int h[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[255 - 8 * lane - i];
    sum += h[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int run = incl - sum, found = -1, before = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (found < 0 && run + h[i] >= need) {
      found = 255 - 8 * lane - i;
      before = run;
    }
    run += h[i];
  }
  const uint32_t who = __ballot_sync(0xffffffffu, found >= 0 && (incl - sum) < need);
  const int src = who ? __ffs(who) - 1 : 0;
  *above = __shfl_sync(0xffffffffu, before, src);
  return __shfl_sync(0xffffffffu, found, src);
}

// One warp per token row: magnitude pruning (radix select of the D/2-th largest
// |v| on 16-bit keys, equal keys kept in index order), bitmap by ballot, kept
// values' sign/high-mantissa and low-mantissa nibbles and pruned raw values in
// order, unary exponent codes at offsets from a warp scan of the code lengths.
__global__ void __launch_bounds__(kEncWarps * 32) kv_encode_kernel(const __grid_constant__ KvEncArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ uint8_t rank_of[256];
  const int D = a.D, K2 = D / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t per_warp = ((size_t)D * 2 + 1024 + (size_t)D / 16 * 8 + (size_t)a.slot_words * 4 + 15) / 16 * 16;
  unsigned char* wb = smem + (size_t)warp * per_warp;
  uint16_t* vals = reinterpret_cast<uint16_t*>(wb);
  int* hist = reinterpret_cast<int*>(wb + (size_t)D * 2);
  uint32_t* sm_w = reinterpret_cast<uint32_t*>(hist + 256);
  uint32_t* lo_w = sm_w + D / 16;
  uint32_t* slot = lo_w + D / 16;
  const uint32_t below = lanemask_lt();

  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    rank_of[(a.cb_words[i >> 2] >> ((i & 3) * 8)) & 0xFFu] = (uint8_t)i;
  if (blockIdx.x == 0 && warp == 0) {
    for (int i = lane; i < 256; i += 32) a.codebook[i] = (uint8_t)((a.cb_words[i >> 2] >> ((i & 3) * 8)) & 0xFFu);
    for (int gi = 0; gi < 7; ++gi)
      for (int64_t q = a.gap_begin[gi] + lane; q < a.gap_end[gi]; q += 32) a.base[q] = 0;
    if (lane == 0) a.rowstart[a.T] = (uint32_t)a.T * (uint32_t)a.slot_words;
  }
  __syncthreads();

  for (int n = blockIdx.x * kEncWarps + warp; n < a.T; n += gridDim.x * kEncWarps) {
    const uint16_t* row = a.v + (size_t)n * a.ld;
    for (int j = lane; j < D; j += 32) vals[j] = row[j];
    for (int i = lane; i < D / 16; i += 32) sm_w[i] = lo_w[i] = 0u;
    for (int i = lane; i < a.slot_words; i += 32) slot[i] = 0u;
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    // ---- radix select: high byte, then low byte among keys with that high byte
    for (int j = lane; j < D; j += 32) atomicAdd(&hist[magnitude_key(vals[j]) >> 8], 1);
    __syncwarp();
    int above1, above0;
    const int d1 = select_digit(hist, K2, &above1);
    __syncwarp();
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int j = lane; j < D; j += 32) {
      const uint32_t k = magnitude_key(vals[j]);
      if ((int)(k >> 8) == d1) atomicAdd(&hist[k & 0xFFu], 1);
    }
    __syncwarp();
    const int d0 = select_digit(hist, K2 - above1, &above0);
    const uint32_t thr = ((uint32_t)d1 << 8) | (uint32_t)d0;
    const int ties_kept = K2 - above1 - above0;  // how many keys equal to thr are kept
    // ---- bitmap, kept nibbles, pruned values and unary codes, 32 columns at a time
    int kb = 0, tb = 0;
    uint32_t bitoff = 0;
    bool overflow = false;
    for (int w = 0; w < D / 32; ++w) {
      const int j = w * 32 + lane;
      const uint32_t b = vals[j];
      const uint32_t k = magnitude_key(b);
      const bool tie = k == thr;
      const uint32_t tball = __ballot_sync(0xffffffffu, tie);
      const bool kept = k > thr || (tie && tb + __popc(tball & below) < ties_kept);
      const uint32_t km = __ballot_sync(0xffffffffu, kept);
      if (lane == 0) a.bitmap[(size_t)n * (D / 32) + w] = km;
      const int kidx = kb + __popc(km & below);
      uint32_t len = 0, r = 0;
      if (kept) {
        const uint32_t sh = (kidx & 7) * 4;
        atomicOr(&sm_w[kidx >> 3], (((b >> 15) << 3) | ((b >> 4) & 7u)) << sh);
        atomicOr(&lo_w[kidx >> 3], (b & 15u) << sh);
        r = rank_of[(b >> 7) & 0xFFu];
        len = r + 1;
      } else {
        a.pruned[(size_t)n * K2 + (j - kidx)] = (uint16_t)b;
      }
      uint32_t incl = len;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (kept) {
        const uint32_t pos = bitoff + incl - len + r;
        if (pos < (uint32_t)a.slot_words * 32u) atomicOr(&slot[pos >> 5], 1u << (pos & 31u));
        else overflow = true;
      }
      bitoff += __shfl_sync(0xffffffffu, incl, 31);
      kb += __popc(km);
      tb += __popc(tball);
    }
    if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicCAS(a.err, 0, (int)QMV_ERR_UNSUPPORTED);
    __syncwarp();
    for (int i = lane; i < D / 16; i += 32) {
      a.signmant[(size_t)n * (D / 16) + i] = sm_w[i];
      a.mlo[(size_t)n * (D / 16) + i] = lo_w[i];
    }
    for (int i = lane; i < a.slot_words; i += 32) a.stream[(size_t)n * a.slot_words + i] = slot[i];
    if (lane == 0) a.rowstart[n] = (uint32_t)n * (uint32_t)a.slot_words;
    __syncwarp();  // the warp's buffers are reused by its next row
  }
}

template <bool TARGET>
int launch_cass(const CassArgs& a, int M, cudaStream_t s) {
  const size_t K = a.K;
  const size_t per_warp = (K / 2 + K / 8 + K / 4 + (TARGET ? K / 4 + K : 0) + 15) / 16 * 16;
  const size_t fixed = (size_t)M * K * 4 + 256;
  const size_t cap = 227 * 1024 - 1024;
  if (fixed + per_warp > cap) return fail(QMV_ERR_UNSUPPORTED, "K=%zu with M=%d does not fit shared memory", K, M);
  const int warps = (int)std::min<size_t>(kCassWarpsMax, (cap - fixed) / per_warp);
  const size_t smem = fixed + per_warp * warps;
  const void* kern = nullptr;
  switch (M) {
#define QMV_CASS_CASE(m) \
  case m: kern = (const void*)cass_kernel<m, TARGET>; break;
    QMV_CASS_CASE(1) QMV_CASS_CASE(2) QMV_CASS_CASE(3) QMV_CASS_CASE(4)
    QMV_CASS_CASE(5) QMV_CASS_CASE(6) QMV_CASS_CASE(7) QMV_CASS_CASE(8)
#undef QMV_CASS_CASE
    default: return fail(QMV_ERR_ARG, "M=%d outside 1..8", M);
  }
  int per_sm = 0;
  int rc = kernel_fit(kern, warps * 32, smem, &per_sm);
  if (rc) return rc;
  const int grid = std::max(1, std::min(sm_count() * per_sm, (a.N + warps - 1) / warps));
  void* args[] = {const_cast<CassArgs*>(&a)};
  cudaError_t e = cudaLaunchKernel(kern, grid, warps * 32, args, smem, s);
  if (e != cudaSuccess) return cuda_fail(e, "cassandra launch");
  return QMV_OK;
}

int check_cass_desc(const qmv_desc* d) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  if (d->abi_version != QMV_ABI_VERSION || d->format != QMV_CASS) return fail(QMV_ERR_ARG, "not a Cassandra descriptor");
  if (d->N <= 0 || d->K <= 0 || d->K % 32) return fail(QMV_ERR_ARG, "N=%lld K=%lld (K must be a multiple of 32)", (long long)d->N, (long long)d->K);
  if (d->N > INT32_MAX / 2 || d->K > (1 << 20)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  const int64_t N = d->N, K = d->K;
  const int64_t want[7] = {N * K / 8, N * K / 4, -1, (N + 1) * 4, 256, N * K, N * K / 4};
  for (int i = 0; i < 7; ++i) {
    if (want[i] >= 0 && d->bytes[i] != want[i]) return fail(QMV_ERR_ARG, "Cassandra section %d has %lld bytes, expected %lld", i, (long long)d->bytes[i], (long long)want[i]);
    if (d->off[i] % 256 || d->off[i] + d->bytes[i] > d->total_bytes) return fail(QMV_ERR_ARG, "Cassandra section %d outside the buffer", i);
  }
  if (d->bytes[2] % 16) return fail(QMV_ERR_ARG, "exponent stream size must be a multiple of 16 bytes");
  if (d->n_symbols < 1 || d->n_symbols > 256) return fail(QMV_ERR_ARG, "n_symbols=%d", d->n_symbols);
  return QMV_OK;
}

int check_cassmx_desc(const qmv_desc* d) {
  if (d->N <= 0 || d->K <= 0 || d->K % 64 || d->group != 32)
    return fail(QMV_ERR_ARG, "N=%lld K=%lld group=%d (K must be a multiple of 64, group 32)", (long long)d->N,
                (long long)d->K, d->group);
  if (d->N > INT32_MAX / 2 || d->K > (1 << 20)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  qmv_desc ref;
  qmv_pack_desc(QMV_CASS_MX, d->N, d->K, 32, &ref);
  for (int i = 0; i < 6; ++i)
    if (ref.off[i] != d->off[i] || ref.bytes[i] != d->bytes[i])
      return fail(QMV_ERR_ARG, "Cassandra-2 section %d does not match the layout of a %lld x %lld matrix", i,
                  (long long)d->N, (long long)d->K);
  return QMV_OK;
}

int run_cass(bool target, const qmv_desc* d, const void* packed, const void* x, int M, int64_t ldx, float* y,
             int64_t ldy, uint16_t* w_out, void* stream) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  const bool mx = d->abi_version == QMV_ABI_VERSION && d->format == QMV_CASS_MX;
  int rc = mx ? check_cassmx_desc(d) : check_cass_desc(d);
  if (rc) return rc;
  if (M < 1 || M > 8) return fail(QMV_ERR_ARG, "M=%d outside 1..8", M);
  if (!packed || !x) return fail(QMV_ERR_ARG, "NULL packed or x");
  if (!aligned16(packed) || !aligned16(x) || (y && !aligned16(y)) || (w_out && !aligned16(w_out)))
    return fail(QMV_ERR_ALIGN, "buffers must be 16-byte aligned");
  if (ldx < d->K || (y && ldy < d->N)) return fail(QMV_ERR_ARG, "ldx < K or ldy < N");
  if (ldx > INT32_MAX || ldy > INT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "leading dimension too large");
  int* err = device_error_word();
  if (!err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  const char* b = static_cast<const char*>(packed);
  if (mx) {
    CassMxArgs m;
    m.bitmap = reinterpret_cast<const uint32_t*>(b + d->off[0]);
    m.gexp = reinterpret_cast<const uint8_t*>(b + d->off[1]);
    m.signs = reinterpret_cast<const uint32_t*>(b + d->off[2]);
    m.dnib = reinterpret_cast<const uint32_t*>(b + d->off[3]);
    m.lnib = reinterpret_cast<const uint32_t*>(b + d->off[4]);
    m.pruned = reinterpret_cast<const uint16_t*>(b + d->off[5]);
    m.x = static_cast<const uint16_t*>(x);
    m.y = y;
    m.w_out = w_out;
    m.N = (int)d->N;
    m.K = (int)d->K;
    m.ldx = (int)ldx;
    m.ldy = (int)(y ? ldy : 0);
    m.err = err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return target ? launch_cassmx<true>(m, M, s) : launch_cassmx<false>(m, M, s);
  }
  CassArgs a;
  a.bitmap = reinterpret_cast<const uint32_t*>(b + d->off[0]);
  a.signmant = reinterpret_cast<const uint32_t*>(b + d->off[1]);
  a.stream = reinterpret_cast<const uint32_t*>(b + d->off[2]);
  a.rowstart = reinterpret_cast<const uint32_t*>(b + d->off[3]);
  a.codebook = reinterpret_cast<const uint8_t*>(b + d->off[4]);
  a.pruned = reinterpret_cast<const uint16_t*>(b + d->off[5]);
  a.mlo = reinterpret_cast<const uint32_t*>(b + d->off[6]);
  a.x = static_cast<const uint16_t*>(x);
  a.y = y;
  a.w_out = w_out;
  a.stream_words = d->bytes[2] / 4;
  a.N = (int)d->N;
  a.K = (int)d->K;
  a.ldx = (int)ldx;
  a.ldy = (int)(y ? ldy : 0);
  a.n_symbols = d->n_symbols;
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return target ? launch_cass<true>(a, M, s) : launch_cass<false>(a, M, s);
}

// ----------------------------------------------------------------------------- host packers

int64_t align256(int64_t n) { return (n + 255) / 256 * 256; }

double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

// Wanda value pruning ("Cassandra", 3.2 step 1): keep[n*K + j] = 1 for the K/2
// largest |w| * ||X[:,j]||_2 of each row (float64; column norms summed over the
// calibration rows in order; equal scores keep the lower column; NaN scores as
// +inf).
void wanda_select(const uint16_t* w, int64_t N, int64_t K, const uint16_t* X, int64_t R, std::vector<uint8_t>& keep) {
  const int64_t K2 = K / 2;
  std::vector<double> c(K, 0.0);
  for (int64_t r = 0; r < R; ++r)
    for (int64_t j = 0; j < K; ++j) {
      const double v = bf16_value(X[r * K + j]);
      c[j] += v * v;
    }
  for (int64_t j = 0; j < K; ++j) c[j] = std::sqrt(c[j]);
  keep.assign((size_t)(N * K), 0);
  std::vector<double> score(K);
  std::vector<int32_t> idx(K);
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = w + n * K;
    for (int64_t j = 0; j < K; ++j) {
      const double s = std::fabs(bf16_value(row[j])) * c[j];
      score[j] = std::isnan(s) ? HUGE_VAL : s;
      idx[j] = (int32_t)j;
    }
    auto before = [&](int32_t a2, int32_t b2) { return score[a2] > score[b2] || (score[a2] == score[b2] && a2 < b2); };
    std::nth_element(idx.begin(), idx.begin() + K2, idx.end(), before);
    for (int64_t i = 0; i < K2; ++i) keep[n * K + idx[i]] = 1;
  }
}

}  // namespace
}  // namespace qmv

using namespace qmv;

extern "C" {

int cass_pack_host(const uint16_t* w, int64_t N, int64_t K, const uint16_t* X, int64_t R, qmv_desc* desc, void* out,
                   int64_t out_capacity) {
  if (!w || !X || !desc) return fail(QMV_ERR_ARG, "NULL w, calibration or desc");
  if (N <= 0 || K <= 0 || K % 32 || R <= 0) return fail(QMV_ERR_ARG, "N=%lld K=%lld R=%lld (K must be a positive multiple of 32)", (long long)N, (long long)K, (long long)R);
  if (N > INT32_MAX / 2 || K > (1 << 20)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  const int64_t K2 = K / 2;
  // 1.-2. Wanda selection per row, then 3. the exponents of the kept values
  std::vector<uint8_t> keep;
  wanda_select(w, N, K, X, R, keep);
  std::vector<uint8_t> ek((size_t)(N * K2));
  std::vector<int64_t> hist(256, 0);
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = w + n * K;
    int64_t k = 0;
    for (int64_t j = 0; j < K; ++j)
      if (keep[n * K + j]) {
        const uint8_t e = (uint8_t)((row[j] >> 7) & 0xFF);
        ek[n * K2 + k++] = e;
        ++hist[e];
      }
  }
  // 4. exponent ranks: count descending, equal counts smaller exponent first
  std::vector<int> order;
  for (int e = 0; e < 256; ++e)
    if (hist[e]) order.push_back(e);
  std::stable_sort(order.begin(), order.end(), [&](int a2, int b2) { return hist[a2] > hist[b2]; });
  std::vector<int> rank_of(256, -1);
  for (size_t r = 0; r < order.size(); ++r) rank_of[order[r]] = (int)r;
  // 5. unary stream length: sum (rank + 1) bits per row, rows padded to 4 words
  std::vector<uint32_t> rowstart((size_t)N + 1, 0);
  for (int64_t n = 0; n < N; ++n) {
    int64_t bits = 0;
    for (int64_t k = 0; k < K2; ++k) bits += rank_of[ek[n * K2 + k]] + 1;
    const int64_t words = ((bits + 31) / 32 + 3) / 4 * 4;
    if ((int64_t)rowstart[n] + words > (int64_t)UINT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "exponent stream too long");
    rowstart[n + 1] = rowstart[n] + (uint32_t)words;
  }
  // layout
  const int64_t sizes[7] = {N * K / 8, N * K / 4, (int64_t)rowstart[N] * 4, (N + 1) * 4, 256, N * K, N * K / 4};
  memset(desc, 0, sizeof(*desc));
  desc->abi_version = QMV_ABI_VERSION;
  desc->format = QMV_CASS;
  desc->N = N;
  desc->K = K;
  desc->group = 0;
  desc->n_symbols = (int32_t)order.size();
  int64_t pos = 0;
  for (int i = 0; i < 7; ++i) {
    desc->off[i] = pos;
    desc->bytes[i] = sizes[i];
    pos = align256(pos + sizes[i]);
  }
  desc->total_bytes = pos;
  if (!out) return QMV_OK;
  if (out_capacity < desc->total_bytes) return fail(QMV_ERR_ARG, "out_capacity %lld < %lld", (long long)out_capacity, (long long)desc->total_bytes);

  unsigned char* o = static_cast<unsigned char*>(out);
  memset(o, 0, (size_t)desc->total_bytes);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(o + desc->off[0]);
  uint32_t* signmant = reinterpret_cast<uint32_t*>(o + desc->off[1]);
  uint32_t* stream = reinterpret_cast<uint32_t*>(o + desc->off[2]);
  uint32_t* rs = reinterpret_cast<uint32_t*>(o + desc->off[3]);
  uint8_t* codebook = o + desc->off[4];
  uint16_t* pruned = reinterpret_cast<uint16_t*>(o + desc->off[5]);
  uint32_t* mlo = reinterpret_cast<uint32_t*>(o + desc->off[6]);
  for (size_t r = 0; r < order.size(); ++r) codebook[r] = (uint8_t)order[r];
  memcpy(rs, rowstart.data(), (size_t)(N + 1) * 4);
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = w + n * K;
    int64_t k = 0, p = 0;
    uint64_t bit = (uint64_t)rowstart[n] * 32;
    for (int64_t j = 0; j < K; ++j) {
      const uint16_t v = row[j];
      if (keep[n * K + j]) {
        bitmap[n * (K / 32) + j / 32] |= 1u << (j % 32);
        const uint32_t S = v >> 15, M = v & 0x7F;
        const int64_t ki = n * K2 + k;
        signmant[ki / 8] |= ((S << 3) | (M >> 4)) << ((ki % 8) * 4);
        mlo[ki / 8] |= (M & 0xF) << ((ki % 8) * 4);
        bit += (uint64_t)rank_of[(v >> 7) & 0xFF];            // rank zeros ...
        stream[bit / 32] |= 1u << (bit % 32);                  // ... then a one
        ++bit;
        ++k;
      } else {
        pruned[n * K2 + p++] = v;
      }
    }
  }
  return QMV_OK;
}

int cass_mx_pack_host(const uint16_t* w, int64_t N, int64_t K, const uint16_t* X, int64_t R, qmv_desc* desc,
                      void* out, int64_t out_capacity) {
  if (!w || !X || !desc) return fail(QMV_ERR_ARG, "NULL w, calibration or desc");
  if (N <= 0 || K <= 0 || K % 64 || R <= 0)
    return fail(QMV_ERR_ARG, "N=%lld K=%lld R=%lld (K must be a positive multiple of 64)", (long long)N, (long long)K, (long long)R);
  if (N > INT32_MAX / 2 || K > (1 << 20)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  int rc = qmv_pack_desc(QMV_CASS_MX, N, K, 32, desc);
  if (rc) return rc;
  if (!out) return QMV_OK;
  if (out_capacity < desc->total_bytes) return fail(QMV_ERR_ARG, "out_capacity %lld < %lld", (long long)out_capacity, (long long)desc->total_bytes);
  std::vector<uint8_t> keep;
  wanda_select(w, N, K, X, R, keep);
  unsigned char* o = static_cast<unsigned char*>(out);
  memset(o, 0, (size_t)desc->total_bytes);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(o + desc->off[0]);
  uint8_t* gexp = o + desc->off[1];
  uint32_t* signs = reinterpret_cast<uint32_t*>(o + desc->off[2]);
  uint32_t* dnib = reinterpret_cast<uint32_t*>(o + desc->off[3]);
  uint32_t* lnib = reinterpret_cast<uint32_t*>(o + desc->off[4]);
  uint16_t* pruned = reinterpret_cast<uint16_t*>(o + desc->off[5]);
  const int64_t K2 = K / 2;
  std::vector<uint16_t> kept((size_t)K2);
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = w + n * K;
    int64_t k = 0, p = 0;
    for (int64_t j = 0; j < K; ++j) {
      if (keep[n * K + j]) {
        bitmap[n * (K / 32) + j / 32] |= 1u << (j % 32);
        kept[k++] = row[j];
      } else {
        pruned[n * K2 + p++] = row[j];
      }
    }
    // groups of 32 kept values share their largest exponent e = max(E, 1)
    for (int64_t g0 = 0; g0 < K2; g0 += 32) {
      int gmax = 1;
      for (int64_t i = g0; i < g0 + 32; ++i) gmax = std::max(gmax, std::max((int)((kept[i] >> 7) & 0xFF), 1));
      gexp[n * (K2 / 32) + g0 / 32] = (uint8_t)gmax;
      for (int64_t i = g0; i < g0 + 32; ++i) {
        const uint32_t v = kept[i], E = (v >> 7) & 0xFF, Mt = v & 0x7F;
        const int e = std::max((int)E, 1);
        const uint32_t sig = (E ? 128u : 0u) + Mt;
        const int sh = gmax - e;
        const uint32_t A = sh < 8 ? sig >> sh : 0u;
        const int64_t ki = n * K2 + i;
        signs[ki / 32] |= (v >> 15) << (ki % 32);
        dnib[ki / 8] |= (A >> 4) << ((ki % 8) * 4);
        lnib[ki / 8] |= (A & 15u) << ((ki % 8) * 4);
      }
    }
  }
  return QMV_OK;
}

int cass_kv_encode(const uint16_t* kv, int64_t T, int64_t D, int64_t ld, const uint8_t* codebook, int64_t slot_words,
                   qmv_desc* desc, void* packed, int64_t capacity, void* stream) {
  if (!codebook || !desc) return fail(QMV_ERR_ARG, "NULL codebook or desc");
  if (T <= 0 || D <= 0 || D % 32 || D > 16384) return fail(QMV_ERR_ARG, "T=%lld D=%lld (D a multiple of 32, at most 16384)", (long long)T, (long long)D);
  if (slot_words <= 0 || slot_words % 4 || slot_words > (int64_t)D * 8) return fail(QMV_ERR_ARG, "slot_words=%lld must be a positive multiple of 4", (long long)slot_words);
  if (T > INT32_MAX / 2 || T * slot_words > (int64_t)UINT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "too many tokens");
  bool seen[256] = {false};
  for (int i = 0; i < 256; ++i) {
    if (seen[codebook[i]]) return fail(QMV_ERR_ARG, "codebook must list each of the 256 exponents once");
    seen[codebook[i]] = true;
  }
  const int64_t sizes[7] = {T * D / 8, T * D / 4, T * slot_words * 4, (T + 1) * 4, 256, T * D, T * D / 4};
  memset(desc, 0, sizeof(*desc));
  desc->abi_version = QMV_ABI_VERSION;
  desc->format = QMV_CASS;
  desc->N = T;
  desc->K = D;
  desc->group = 0;
  desc->n_symbols = 256;
  int64_t pos = 0;
  for (int i = 0; i < 7; ++i) {
    desc->off[i] = pos;
    desc->bytes[i] = sizes[i];
    pos = align256(pos + sizes[i]);
  }
  desc->total_bytes = pos;
  if (!packed) return QMV_OK;
  if (!kv) return fail(QMV_ERR_ARG, "NULL kv");
  if (capacity < desc->total_bytes) return fail(QMV_ERR_ARG, "capacity %lld < %lld", (long long)capacity, (long long)desc->total_bytes);
  if (!aligned16(kv) || !aligned16(packed)) return fail(QMV_ERR_ALIGN, "kv and packed must be 16-byte aligned");
  if (ld < D || ld % 8) return fail(QMV_ERR_ARG, "ld=%lld must be >= D and a multiple of 8", (long long)ld);
  int* err = device_error_word();
  if (!err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  unsigned char* b = static_cast<unsigned char*>(packed);
  KvEncArgs a;
  a.v = kv;
  a.ld = ld;
  a.T = (int)T;
  a.D = (int)D;
  a.slot_words = (int)slot_words;
  a.bitmap = reinterpret_cast<uint32_t*>(b + desc->off[0]);
  a.signmant = reinterpret_cast<uint32_t*>(b + desc->off[1]);
  a.stream = reinterpret_cast<uint32_t*>(b + desc->off[2]);
  a.rowstart = reinterpret_cast<uint32_t*>(b + desc->off[3]);
  a.codebook = b + desc->off[4];
  a.pruned = reinterpret_cast<uint16_t*>(b + desc->off[5]);
  a.mlo = reinterpret_cast<uint32_t*>(b + desc->off[6]);
  a.base = b;
  for (int i = 0; i < 7; ++i) {
    a.gap_begin[i] = desc->off[i] + desc->bytes[i];
    a.gap_end[i] = i + 1 < 7 ? desc->off[i + 1] : desc->total_bytes;
  }
  for (int i = 0; i < 64; ++i)
    a.cb_words[i] = (uint32_t)codebook[4 * i] | ((uint32_t)codebook[4 * i + 1] << 8) | ((uint32_t)codebook[4 * i + 2] << 16) |
                    ((uint32_t)codebook[4 * i + 3] << 24);
  a.err = err;
  const size_t per_warp = ((size_t)D * 2 + 1024 + (size_t)D / 16 * 8 + (size_t)slot_words * 4 + 15) / 16 * 16;
  const size_t smem = per_warp * kEncWarps;
  if (smem > 227 * 1024 - 1024) return fail(QMV_ERR_UNSUPPORTED, "D=%lld with slot_words=%lld does not fit shared memory", (long long)D, (long long)slot_words);
  int per_sm = 0;
  int rc = kernel_fit((const void*)kv_encode_kernel, kEncWarps * 32, smem, &per_sm);
  if (rc) return rc;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)sm_count() * per_sm, (T + kEncWarps - 1) / kEncWarps));
  kv_encode_kernel<<<grid, kEncWarps * 32, smem, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kv encode launch");
  return QMV_OK;
}

int cass_decode_draft(const qmv_desc* desc, const void* packed, const void* x_bf16, int M, int64_t ldx, float* y,
                      int64_t ldy, uint16_t* w_draft, void* stream) {
  return run_cass(false, desc, packed, x_bf16, M, ldx, y, ldy, w_draft, stream);
}

int cass_reconstruct(const qmv_desc* desc, const void* packed, const void* x_bf16, int M, int64_t ldx, float* y,
                     int64_t ldy, uint16_t* w_out, void* stream) {
  return run_cass(true, desc, packed, x_bf16, M, ldx, y, ldy, w_out, stream);
}

}  // extern "C"
