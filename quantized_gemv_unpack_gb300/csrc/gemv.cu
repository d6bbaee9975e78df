// Fused dequantize-and-matvec for block-128 ternary and group-128 INT4 weights.
//
// One persistent launch walks a table of matvecs (one GEMV, the q|k|v group of
// a layer, or a whole decode stack). Work is cut into tiles of 8*RW rows;
// CTA c takes tiles c, c + gridDim.x, ... Each warp owns RW rows of a tile and
// streams them along K: per step a lane reads 8 bytes of codes per row
// (32 ternary or 16 INT4 weights) with a non-allocating 64-bit load and the
// fp16 scale of the block they belong to.
//
// Activations are staged once per (x, chunk) in shared memory as fp16 pairs
// in exactly the order a lane consumes them, after scaling the chunk by a
// power of two so its largest magnitude lies in [2^9, 2^10) (ternary) or
// [2^8, 2^9) (INT4); the scale is undone in fp32.
//
// Decode, per 32-bit code word, without lookup tables:
//  * ternary: the low half holds even columns, the high half odd columns, so a
//    word gives eight (even, odd) column pairs. Shifting pair i's two 2-bit
//    codes to bits 9-10 and 25-26 and computing (t & 0x06000600) ^ 0x3C003C00
//    yields two fp16 values v = 1 + q/2 (code 00 -> 1.0, 01 -> 1.5, 10 -> 0.5):
//    bit 9 is the mantissa MSB (+0.5), bit 10 the exponent LSB (halves 1.0).
//    Then sum_k v_k x_k = sum_k x_k + (1/2) sum_k q_k x_k, and the fp16
//    accumulator is seeded with -sum x over the lane's columns (computed once
//    per staged chunk), leaving (1/2) sum q x; the factor 2 is applied at the end.
//  * INT4: (t & 0x000F000F) ^ 0x64086408 maps a two's-complement nibble q to
//    the fp16 integer 1032 + q (1024 + offset-binary nibble); subtracting 1032
//    gives q exactly, which is then multiplied into the fp16 accumulator.
// Per row and lane step the fp16 pair accumulator is widened to fp32, scaled
// by the block's fp16 scale and added to an fp32 sum; warp shuffles reduce
// the 32 lanes at the end of the tile.
#include <cstring>

#include "qmv_internal.cuh"

namespace qmv {
namespace {

template <int FMT>
struct Fmt;
template <>
struct Fmt<QMV_TERNARY2> {
  static constexpr int KPL = 32;      // columns per lane per step (one 8-byte load)
  static constexpr int PAIRS = 8;     // column pairs per 32-bit word
  static constexpr int COLS_PER_WORD = 16;
  static constexpr int XLOG2 = 9;     // staged |x| max in [2^9, 2^10)
};
template <>
struct Fmt<QMV_INT4> {
  static constexpr int KPL = 16;
  static constexpr int PAIRS = 4;
  static constexpr int COLS_PER_WORD = 8;
  static constexpr int XLOG2 = 8;
};

__host__ __device__ constexpr int rows_per_warp(int mt) { return mt <= 2 ? 4 : (mt <= 4 ? 2 : 1); }

__device__ __forceinline__ uint2 ld_stream_u2(const uint32_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
__device__ __forceinline__ float bf16_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ int find_task(const GemvBatch& b, int tile) {
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// power of two 2^e as a float, e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

template <int FMT>
__device__ __forceinline__ __half2 decode_pair(uint32_t w, int i) {
  if constexpr (FMT == QMV_TERNARY2) {
    // pair i: even column code at bits 2i..2i+1, odd column code at 16+2i..17+2i
    uint32_t t = (i <= 4) ? (w << (9 - 2 * i)) : (w >> (2 * i - 9));
    return as_h2((t & 0x06000600u) ^ 0x3C003C00u);
  } else {
    uint32_t t = w >> (4 * i);
    __half2 v = as_h2((t & 0x000F000Fu) ^ 0x64086408u);
    return __hsub2(v, __floats2half2_rn(1032.f, 1032.f));
  }
}

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvBatch b) {
  using F = Fmt<FMT>;
  constexpr int KPL = F::KPL;
  constexpr int STEP = 32 * KPL;          // columns per warp step
  constexpr int J = KPL / 8;              // 16-byte activation pieces per lane step
  constexpr int RW = rows_per_warp(MT);
  constexpr int ROWS = (kThreads / 32) * RW;
  constexpr bool TERN = FMT == QMV_TERNARY2;

  extern __shared__ __align__(16) unsigned char smem[];
  const int KC = b.kc;
  const int S = KC / STEP;
  uint4* xs = reinterpret_cast<uint4*>(smem);                        // [MT][S][J][32]
  __half2* negs = reinterpret_cast<__half2*>(xs + (size_t)MT * S * J * 32);  // [MT][S][32]
  __shared__ float s_red[kThreads / 32][MT];
  __shared__ float s_xinv[MT];
  __shared__ float s_xscale[MT];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const uint16_t* staged_x = nullptr;
  int staged_c = -1;
  int staged_K = -1;

  for (int tile = blockIdx.x; tile < b.n_tiles; tile += gridDim.x) {
    const int ti = find_task(b, tile);
    const GemvTask& T = b.t[ti];
    const int K = T.K;
    const int KW = K / F::COLS_PER_WORD;
    const int KB = K / 128;
    const int rbase = (tile - T.tile0) * ROWS + warp * RW;
    const int nchunks = (K + KC - 1) / KC;

    float acc[RW][MT];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    for (int c = 0; c < nchunks; ++c) {
      const int kc0 = c * KC;
      const int kcn = min(KC, K - kc0);

      if (T.x != staged_x || c != staged_c || K != staged_K || nchunks > 1) {
        // ---- stage activations of this chunk (all threads of the CTA)
        __syncthreads();
        const int ngroups = kcn / 8;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float mx = 0.f;
          const uint16_t* xr = T.x + (size_t)m * T.ldx + kc0;
          for (int g = tid; g < ngroups; g += kThreads) {
            uint4 raw = *reinterpret_cast<const uint4*>(xr + g * 8);
            uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              mx = fmaxf(mx, fabsf(bf16_to_f32(wv[q] & 0xFFFFu)));
              mx = fmaxf(mx, fabsf(bf16_to_f32(wv[q] >> 16)));
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) s_red[warp][m] = mx;
        }
        __syncthreads();
        if (tid < MT) {
          float mx = 0.f;
#pragma unroll
          for (int w = 0; w < kThreads / 32; ++w) mx = fmaxf(mx, s_red[w][tid]);
          int e = 0;
          if (mx > 0.f && mx <= 3.4e38f) {
            int ex;
            frexpf(mx, &ex);                         // mx = f * 2^ex, f in [0.5, 1)
            e = F::XLOG2 - (ex - 1);
            e = max(-120, min(120, e));
          }
          s_xscale[tid] = exp2i(e);
          s_xinv[tid] = exp2i(-e);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float xsc = s_xscale[m];
          const uint16_t* xr = T.x + (size_t)m * T.ldx + kc0;
          for (int g = tid; g < ngroups; g += kThreads) {
            uint4 raw = *reinterpret_cast<const uint4*>(xr + g * 8);
            uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t hv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              __half2 h = __floats2half2_rn(bf16_to_f32(wv[q] & 0xFFFFu) * xsc, bf16_to_f32(wv[q] >> 16) * xsc);
              hv[q] = *reinterpret_cast<uint32_t*>(&h);
            }
            const int k = g * 8;
            const int s = k / STEP;
            const int l = (k % STEP) / KPL;
            const int j = (k % KPL) / 8;
            xs[(((size_t)m * S + s) * J + j) * 32 + l] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          }
        }
        if constexpr (TERN) {
          __syncthreads();
          for (int g = tid; g < MT * S * 32; g += kThreads) {
            const int m = g / (S * 32);
            const int s = (g / 32) % S;
            const int l = g % 32;
            float se = 0.f, so = 0.f;
            if (s * STEP + l * KPL < kcn) {
#pragma unroll
              for (int j = 0; j < J; ++j) {
                uint4 p = xs[(((size_t)m * S + s) * J + j) * 32 + l];
                uint32_t pv[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float2 f = __half22float2(as_h2(pv[q]));
                  se += f.x;
                  so += f.y;
                }
              }
            }
            negs[g] = __floats2half2_rn(-se, -so);
          }
        }
        __syncthreads();
        staged_x = T.x;
        staged_c = c;
        staged_K = K;
      }

      // ---- stream the rows of this warp over the chunk
      float xinv[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) xinv[m] = s_xinv[m];
      const int nsteps = (kcn + STEP - 1) / STEP;

      uint2 cw_n[RW];
      uint16_t sc_n[RW];
      auto load_step = [&](int s, uint2* cw, uint16_t* sc) {
        const int kl = s * STEP + lane * KPL;
        const int k0 = kc0 + kl;
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          const int row = rbase + r;
          if (row < T.N && kl < kcn) {
            cw[r] = ld_stream_u2(T.codes + (size_t)row * KW + k0 / F::COLS_PER_WORD);
            sc[r] = __ldg(reinterpret_cast<const unsigned short*>(T.scales) + (size_t)row * KB + k0 / 128);
          } else {
            cw[r] = make_uint2(0u, 0u);
            sc[r] = 0;
          }
        }
      };
      load_step(0, cw_n, sc_n);

      for (int s = 0; s < nsteps; ++s) {
        uint2 cw[RW];
        uint16_t sc[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          cw[r] = cw_n[r];
          sc[r] = sc_n[r];
        }
        if (s + 1 < nsteps) load_step(s + 1, cw_n, sc_n);
        const int kl = s * STEP + lane * KPL;
        if (kl >= kcn) continue;

        __half2 a2[RW][MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          __half2 init = TERN ? negs[((size_t)m * S + s) * 32 + lane] : __floats2half2_rn(0.f, 0.f);
#pragma unroll
          for (int r = 0; r < RW; ++r) a2[r][m] = init;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          constexpr int JW = J / 2;     // pieces per word
          uint4 xw[MT][JW];
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < JW; ++j) xw[m][j] = xs[(((size_t)m * S + s) * J + h * JW + j) * 32 + lane];
#pragma unroll
          for (int r = 0; r < RW; ++r) {
            const uint32_t w = h ? cw[r].y : cw[r].x;
#pragma unroll
            for (int i = 0; i < F::PAIRS; ++i) {
              const __half2 v = decode_pair<FMT>(w, i);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint4 p = xw[m][i / 4];
                const uint32_t pv = (i % 4 == 0) ? p.x : (i % 4 == 1) ? p.y : (i % 4 == 2) ? p.z : p.w;
                a2[r][m] = __hfma2(v, as_h2(pv), a2[r][m]);
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          const float scf = __half2float(__ushort_as_half(sc[r]));
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float2 f = __half22float2(a2[r][m]);
            acc[r][m] = fmaf(f.x + f.y, scf * xinv[m], acc[r][m]);
          }
        }
      }
    }

    // ---- reduce over lanes, write y
    constexpr float kFactor = TERN ? 2.f : 1.f;
#pragma unroll
    for (int r = 0; r < RW; ++r) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int row = rbase + r;
        if (lane == 0 && row < T.N) T.y[(size_t)m * T.ldy + row] = kFactor * v;
      }
    }
  }
}

template <int FMT, int MT>
int launch_t(GemvBatch& b, int max_K, cudaStream_t s) {
  constexpr int KPL = Fmt<FMT>::KPL;
  constexpr int STEP = 32 * KPL;
  // activation chunk: as much of K as fits a ~112 KB budget, in whole warp steps
  int kc_cap = (57344 / MT) / STEP * STEP;
  int kc = ((max_K + STEP - 1) / STEP) * STEP;
  if (kc > kc_cap) kc = kc_cap;
  b.kc = kc;
  const size_t S = kc / STEP;
  size_t smem = (size_t)MT * kc * 2 + (FMT == QMV_TERNARY2 ? (size_t)MT * S * 32 * 4 : 0);
  auto kern = gemv_kernel<FMT, MT>;
  int per_sm = 0;
  int rc = kernel_fit((const void*)kern, kThreads, smem, &per_sm);
  if (rc != QMV_OK) return rc;
  int grid = sm_count() * per_sm;
  if (grid > b.n_tiles) grid = b.n_tiles;
  kern<<<grid, kThreads, smem, s>>>(b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
  return QMV_OK;
}

template <int FMT>
int launch_fmt(GemvBatch& b, int M, int max_K, cudaStream_t s) {
  switch (M) {
    case 1: return launch_t<FMT, 1>(b, max_K, s);
    case 2: return launch_t<FMT, 2>(b, max_K, s);
    case 3: return launch_t<FMT, 3>(b, max_K, s);
    case 4: return launch_t<FMT, 4>(b, max_K, s);
    case 5: return launch_t<FMT, 5>(b, max_K, s);
    case 6: return launch_t<FMT, 6>(b, max_K, s);
    case 7: return launch_t<FMT, 7>(b, max_K, s);
    case 8: return launch_t<FMT, 8>(b, max_K, s);
    default: return fail(QMV_ERR_ARG, "M=%d outside 1..8 for one launch", M);
  }
}

}  // namespace

int gemv_rows_per_tile(int M) { return (kThreads / 32) * rows_per_warp(M); }

int launch_gemv(int format, GemvBatch& b, int M, int max_K, cudaStream_t s) {
  if (format == QMV_TERNARY2) return launch_fmt<QMV_TERNARY2>(b, M, max_K, s);
  if (format == QMV_INT4) return launch_fmt<QMV_INT4>(b, M, max_K, s);
  return fail(QMV_ERR_UNSUPPORTED, "format %d has no matvec kernel", format);
}

}  // namespace qmv
