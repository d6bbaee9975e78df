// Building blocks of the fused dequantize-and-matvec kernels, shared by the
// persistent matvec batch (gemv.cu) and the MoE expert kernels (moe.cu): the
// packed formats' decode, the activation staging and the one-step decode of a
// warp's rows from a shared-memory slot. The design notes are in gemv.cu.
#pragma once

#include "qmv_internal.cuh"

namespace qmv {
namespace core {

constexpr int kBlocksPerStepHost = 8;  // 128-column blocks per 1024-column step (kBlocksPerStep)

template <int FMT>
struct Fmt;
template <>
struct Fmt<QMV_TERNARY2> {
  static constexpr int WPB = 8;    // 32-bit code words per 128-column block
  static constexpr int PPW = 8;    // column pairs per word
  static constexpr int CPW = 16;   // columns per word
  static constexpr int JW = 2;     // 16-byte activation pieces per word
  // staged |x| max in [2^13, 2^14): a chain of four products |q/2 x| <= 2^13
  // stays below 2^15, and values down to 2^-29 of the largest stay exact in fp16
  static constexpr int XLOG2 = 13;
  static constexpr uint32_t MASK = 0x06000600u, BASE = 0x3C003C00u;
};
template <>
struct Fmt<QMV_INT4> {
  static constexpr int WPB = 16;
  static constexpr int PPW = 4;
  static constexpr int CPW = 8;
  static constexpr int JW = 1;
  // staged |x| max in [2^10, 2^11): a chain of four products |q x| <= 7 * 2^11
  // stays below the fp16 maximum (65504)
  static constexpr int XLOG2 = 10;
  static constexpr uint32_t MASK = 0x000F000Fu, BASE = 0x64086408u;
};

// fp16 accumulation chains of kChainPairs column pairs: each chain starts from
// an exact product and takes three more fp16 FMAs, then its two halves are
// added into an fp32 block sum (mixed-precision adds). With exact products the
// chain's rounding error is at most 3 * 2^-11 of the sum of its |terms|, which
// keeps every row within 1.5e-3 of sum_k |w_hat_k x_k|.
constexpr int kChainPairs = 4;

constexpr int kGroups = 4;            // lane groups (rows of a row quad)
constexpr int kBlocksPerStep = kBlocksPerStepHost;  // lanes per row
constexpr int kStep = kBlocksPerStep * 128;
constexpr int kSlots = 2;             // ring slots per decode warp
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr uint64_t kWaitNs = 2000000000ull;  // a wait not done after 2 s is declared lost

// (a & b) ^ c as one logic op
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// a * m on the integer-multiply unit (m a run-time power of two: a left shift)
__device__ __forceinline__ uint32_t mul_lo(uint32_t a, uint32_t m) {
  uint32_t d;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(m));
  return d;
}
// shifts by a run-time amount on the shift unit
__device__ __forceinline__ uint32_t shl_r(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(s));
  return d;
}
__device__ __forceinline__ uint32_t shr_r(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("shr.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(s));
  return d;
}

// decode constants held in registers for the whole kernel
struct DecodeK {
  uint32_t mask, base;
  uint32_t m9, m7, m5, m1;  // 2^9, 2^7, 2^5, 2^1
  uint32_t s1, s3, s5;      // shift amounts 1, 3, 5 (INT4: 4, 8, 12)
};

__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ float bf16_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }
// 2^e as a float, e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// fp32 a + the two fp16 halves of h (mixed-precision adds, exact widening)
__device__ __forceinline__ float add_h2_f32(float a, __half2 h) {
  float d;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 t;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 t, lo, %2;\n\tadd.rn.f32.f16 %0, hi, t;\n\t}"
      : "=f"(d)
      : "r"(*reinterpret_cast<const uint32_t*>(&h)), "f"(a));
  return d;
}

// The two weights of column pair i of code word w as fp16, exactly: ternary
// q/2 (code 00 -> 0, 01 -> +1/2, 10 -> -1/2), INT4 q.
template <int FMT>
__device__ __forceinline__ __half2 decode_pair(uint32_t w, int i, const DecodeK& k) {
  if constexpr (FMT == QMV_TERNARY2) {
    // pair i: even column code at bits 2i..2i+1, odd column code at 16+2i..17+2i;
    // shift both to bits 9-10 / 25-26, where (t & mask) ^ base gives v = 1 + q/2
    uint32_t t;
    switch (i) {
      case 0: t = mul_lo(w, k.m9); break;
      case 1: t = mul_lo(w, k.m7); break;
      case 2: t = mul_lo(w, k.m5); break;
      case 3: t = shl_r(w, k.s3); break;
      case 4: t = mul_lo(w, k.m1); break;
      case 5: t = shr_r(w, k.s1); break;
      case 6: t = shr_r(w, k.s3); break;
      default: t = shr_r(w, k.s5); break;
    }
    return __hsub2(as_h2(and_xor(t, k.mask, k.base)), __floats2half2_rn(1.f, 1.f));
  } else {
    const uint32_t t = i == 0 ? w : shr_r(w, i == 1 ? k.s1 : (i == 2 ? k.s3 : k.s5));
    return __hsub2(as_h2(and_xor(t, k.mask, k.base)), __floats2half2_rn(1032.f, 1032.f));
  }
}

// ---- mbarrier and bulk-copy helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false (and QMV_ERR_TIMEOUT in the device error word) if the
// phase does not complete within limit_ns. Once the error word holds a timeout,
// later waits give up after a few hundred polls, so a launch that lost a
// barrier ends quickly instead of timing out wait after wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t polls = 1;; ++polls) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((polls & 255u) == 0u &&
        (global_ns() - t0 > limit_ns || *reinterpret_cast<volatile int*>(err) == (int)QMV_ERR_TIMEOUT))
      break;
  }
  atomicCAS(err, 0, (int)QMV_ERR_TIMEOUT);
  return false;
}
// Testing hook (QMV_FLAG_TEST_WAIT_TIMEOUT): before any copy is issued, thread
// 0 waits on a barrier that nothing completes, with a limit of `us`
// microseconds, so the wait gives up and records QMV_ERR_TIMEOUT; true means
// the kernel must return at once (nothing is in flight). Called by every
// thread of the CTA.
__device__ __forceinline__ bool test_wait_times_out(int* err, uint32_t us) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int gave_up;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    gave_up = mbar_wait(&bar, 0u, err, (uint64_t)us * 1000ull) ? 0 : 1;
  }
  __syncthreads();
  return gave_up != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

template <int FMT, int RPW>
struct Geometry {
  static constexpr int BLOCK_BYTES = Fmt<FMT>::WPB * 4;
  static constexpr int ROW_STEP_BYTES = kBlocksPerStep * BLOCK_BYTES;   // one step of one row
  static constexpr int SLOT = RPW * ROW_STEP_BYTES;
  static constexpr int RING = kConsumerWarps * kSlots * SLOT;
  static constexpr int BARS = kConsumerWarps * kSlots * 8;
  static constexpr int TILE_ROWS = kConsumerWarps * RPW;
};


// Activation sources for staging. load8(m, k, v) returns the 8 consecutive
// activations k..k+7 (chunk-relative) of activation row m as floats.
struct Bf16Rows {  // x[m][ldx], bf16
  const uint16_t* x;
  int ldx, kc0;
  __device__ __forceinline__ void load8(int m, int k, float v[8]) const {
    const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)m * ldx + kc0 + k);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t wv = word_of(raw, e);
      v[2 * e] = bf16_to_f32(wv & 0xFFFFu);
      v[2 * e + 1] = bf16_to_f32(wv >> 16);
    }
  }
};

// Stage columns [kc0, kc0 + kcn) of MT activation rows into shared memory: fp16
// pairs in the order a lane consumes them, scaled by a power of two per row so
// the largest magnitude lands in [2^XLOG2, 2^(XLOG2+1)). bf16 values have 8
// significant bits, so the scaled values are exact in fp16 down to 2^-17
// (subnormal spacing 2^-24). Called by every thread of the CTA (NT threads);
// begins and ends with a CTA barrier.
template <int FMT, int MT, int NT, class Src>
__device__ void stage_chunk(const Src& src, int kcn, int S, uint4* xs, float (*s_red)[MT], float* s_xscale,
                            float* s_xinv) {
  using F = Fmt<FMT>;
  constexpr int WPB = F::WPB;
  constexpr int JW = F::JW;
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ngroups = kcn / 8;
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float mx = 0.f;
    for (int q = tid; q < ngroups; q += NT) {
      float v[8];
      src.load8(m, q * 8, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp][m] = mx;
  }
  __syncthreads();
  if (tid < MT) {
    float mx = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, s_red[w][tid]);
    int e = 0;
    if (mx > 0.f && mx <= 3.4e38f) {
      int ex;
      frexpf(mx, &ex);  // mx = f * 2^ex, f in [0.5, 1)
      e = max(-120, min(120, F::XLOG2 - (ex - 1)));
    }
    s_xscale[tid] = exp2i(e);
    s_xinv[tid] = exp2i(-e);
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const float xsc = s_xscale[m];
    for (int q = tid; q < ngroups; q += NT) {
      float v[8];
      src.load8(m, q * 8, v);
      uint32_t hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __half2 h = __floats2half2_rn(v[2 * e] * xsc, v[2 * e + 1] * xsc);
        hv[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      const int k = q * 8;
      const int blk = k / 128, cc = k % 128;
      const int s = blk / kBlocksPerStep, pp = blk % kBlocksPerStep;
      const int h = cc / F::CPW, j = (cc % F::CPW) / 8;
      xs[((((size_t)m * S + s) * WPB + h) * JW + j) * 8 + pp] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
  }
  __syncthreads();
}

// Decode one step (up to 8 blocks) of RQ row quads held in a shared-memory
// slot and accumulate sum_k w_hat x per row and activation row into accc
// (fp32, in units of the block scale times the staged activation scale; for
// ternary half of that, since the decode gives q/2). sb points at the slot plus
// this lane's block; rows are row_bytes apart. The 16-byte activation piece j
// of word h holds the word's column pairs 4j .. 4j+3, i.e. one chain.
template <int FMT, int MT, int RQ>
__device__ __forceinline__ void decode_step(const unsigned char* sb, int row_bytes, const uint4* xs, int S, int s,
                                            int g, int p, const DecodeK& dk, const unsigned short (&sc)[RQ],
                                            float (&accc)[RQ][MT]) {
  using F = Fmt<FMT>;
  constexpr int WPB = F::WPB;
  constexpr int JW = F::JW;
  static_assert(F::PPW == JW * kChainPairs, "one chain per 16-byte activation piece");
  uint4 cw[RQ][WPB / 4];
#pragma unroll
  for (int r = 0; r < RQ; ++r)
#pragma unroll
    for (int u = 0; u < WPB / 4; ++u)
      cw[r][u] = *reinterpret_cast<const uint4*>(sb + (r * kGroups + g) * row_bytes + u * 16);
  float bsum[RQ][MT];
#pragma unroll
  for (int r = 0; r < RQ; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) bsum[r][m] = 0.f;
  auto xload = [&](int m, int h, int j) { return xs[((((size_t)m * S + s) * WPB + h) * JW + j) * 8 + p]; };
  // one chain: four exact products summed in fp16, then widened into the block sum
  auto chain = [&](const __half2 (&v)[kChainPairs], const uint4& xw, float& acc) {
    __half2 c = __hmul2(v[0], as_h2(xw.x));
    c = __hfma2(v[1], as_h2(xw.y), c);
    c = __hfma2(v[2], as_h2(xw.z), c);
    c = __hfma2(v[3], as_h2(xw.w), c);
    acc = add_h2_f32(acc, c);
  };
#pragma unroll
  for (int h = 0; h < WPB; ++h) {
    if constexpr (RQ == 1) {
      // one row: decode the word once, then stream each activation row through it
      const uint32_t w = word_of(cw[0][h / 4], h % 4);
#pragma unroll
      for (int j = 0; j < JW; ++j) {
        __half2 v[kChainPairs];
#pragma unroll
        for (int i = 0; i < kChainPairs; ++i) v[i] = decode_pair<FMT>(w, j * kChainPairs + i, dk);
#pragma unroll
        for (int m = 0; m < MT; ++m) chain(v, xload(m, h, j), bsum[0][m]);
      }
    } else {
      // several rows share each activation load
#pragma unroll
      for (int j = 0; j < JW; ++j) {
        uint4 xw[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) xw[m] = xload(m, h, j);
#pragma unroll
        for (int r = 0; r < RQ; ++r) {
          const uint32_t w = word_of(cw[r][h / 4], h % 4);
          __half2 v[kChainPairs];
#pragma unroll
          for (int i = 0; i < kChainPairs; ++i) v[i] = decode_pair<FMT>(w, j * kChainPairs + i, dk);
#pragma unroll
          for (int m = 0; m < MT; ++m) chain(v, xw[m], bsum[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RQ; ++r) {
    const float scf = __half2float(__ushort_as_half(sc[r]));
#pragma unroll
    for (int m = 0; m < MT; ++m) accc[r][m] = fmaf(bsum[r][m], scf, accc[r][m]);
  }
}

// Fill the decode constants of a format into magic[0..9] (see DecodeK).
template <int FMT>
inline void fill_magic(uint32_t* magic) {
  magic[0] = Fmt<FMT>::MASK;
  magic[1] = Fmt<FMT>::BASE;
  magic[2] = 1u << 9;
  magic[3] = 1u << 7;
  magic[4] = 1u << 5;
  magic[5] = 1u << 1;
  const bool tern = FMT == QMV_TERNARY2;
  magic[6] = tern ? 1 : 4;
  magic[7] = tern ? 3 : 8;
  magic[8] = tern ? 5 : 12;
  magic[9] = 0;
}

__device__ __forceinline__ DecodeK load_decode_k(const uint32_t* m) {
  return DecodeK{m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], m[8]};
}

}  // namespace core
}  // namespace qmv
