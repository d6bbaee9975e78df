// Offline quantize-and-pack kernels (ternary, INT4) and the decode-to-int8
// kernel used for bit-exact checks of the packed stream.
//
// One thread owns one 128-column block of one row: it sums |w| in float64 in
// column order, divides in float64 and rounds half to even, so the codes and
// the fp16 scales are fully determined by the input (no reduction-order
// freedom). The float64 -> fp16 rounding is done on the bit patterns,
// nearest-even in one step, from the IEEE-754 binary16 definition.
#include "lut.cuh"

namespace qmv {
namespace {

// binary16 bits of a float64, round to nearest, ties to even (no float32 detour)
__device__ uint16_t f64_to_f16_rne(double d) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(d);
  const uint32_t sign = (uint32_t)(b >> 63) << 15;
  const int e = (int)((b >> 52) & 0x7FF);
  const unsigned long long f = b & ((1ull << 52) - 1);
  if (e == 0x7FF) return (uint16_t)(sign | (f ? 0x7E00u : 0x7C00u));
  const int eu = e ? e - 1023 : -1022;                   // value = sig * 2^(eu - 52)
  const unsigned long long sig = e ? (f | (1ull << 52)) : f;
  const int shift = eu >= -14 ? 42 : 28 - eu;            // to units of the fp16 ulp
  if (shift >= 64) return (uint16_t)sign;
  unsigned long long kept = sig >> shift;
  const unsigned long long rem = sig & ((1ull << shift) - 1);
  const unsigned long long half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (kept & 1ull))) ++kept;
  unsigned long long enc = eu >= -14 ? ((unsigned long long)(eu + 14) << 10) + kept : kept;
  if (enc >= 0x7C00ull) enc = 0x7C00ull;
  return (uint16_t)(sign | (uint32_t)enc);
}

// Word offset of block b of row n in the row-group record layout of the codes
// section: groups of 16 rows, steps of 8 blocks, each record row-major.
__device__ __forceinline__ int64_t record_word(int64_t n, int64_t b, int64_t K, int block_words) {
  const int64_t KB = K / 128;
  const int64_t g = n / 16, r = n % 16, st = b / 8, j = b % 8;
  const int64_t nbk = KB - st * 8 < 8 ? KB - st * 8 : 8;
  return ((g * 16 * KB + st * 16 * 8) + r * nbk + j) * block_words;
}

// Byte offset of byte t of (row n, block b) in the lookup layout's codes
// section (QMV_TERNARY2_LUT): 1 KB records of (block, 32-row group), each
// row's 32 bytes rotated by n % 32 (byte t holds column group (t + n) % 32).
__host__ __device__ __forceinline__ int64_t lut_byte(int64_t n, int64_t b, int t, int64_t NG) {
  return (b * NG + n / 32) * 1024 + (t / 16) * 512 + (n % 32) * 16 + t % 16;
}

// Byte offset of position t (0..63) of (row n, block b) in the INT4 lookup
// layout's codes section (QMV_INT4_LUT): 2 KB records of (block, 32-row group).
__host__ __device__ __forceinline__ int64_t lut4_byte(int64_t n, int64_t b, int t, int64_t NG) {
  return (b * NG + n / 32) * 2048 + (t / 16) * 512 + (n % 32) * 16 + t % 16;
}

template <bool LUT>
__global__ void pack_ternary_kernel(const float* __restrict__ w, int64_t N, int64_t K, uint32_t* __restrict__ codes,
                                    uint16_t* __restrict__ scales) {
  const int64_t nb = K / 128;
  const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= N * nb) return;
  const int64_t n = blk / nb, b = blk % nb;
  const float4* src = reinterpret_cast<const float4*>(w + n * K + b * 128);
  double acc = 0.0;
  for (int i = 0; i < 32; ++i) {
    const float4 v = src[i];
    acc += fabs((double)v.x);
    acc += fabs((double)v.y);
    acc += fabs((double)v.z);
    acc += fabs((double)v.w);
  }
  const double s = acc / 128.0 + 1e-8;
  uint32_t words[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) words[j] = 0u;
  for (int i = 0; i < 32; ++i) {
    const float4 v = src[i];
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int k = i * 4 + c;
      const double r = rint((double)vv[c] / s);
      const uint32_t code = r >= 1.0 ? 1u : (r <= -1.0 ? 2u : 0u);
      const int rr = k & 15;
      const int pos = (rr & 1) ? 15 + rr : rr;
      words[k >> 4] |= code << pos;
    }
  }
  if constexpr (LUT) {
    // group c (columns 4c..4c+3) as one byte, column 4c + i at bits 2i
    uint32_t gb[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      uint32_t v = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = 4 * c + i, rr = k & 15;
        const int pos = (rr & 1) ? 15 + rr : rr;
        v |= ((words[k >> 4] >> pos) & 3u) << (2 * i);
      }
      gb[c] = v;
    }
    const int64_t NG = (N + 31) / 32;
    const int rot = (int)(n % 32);
    uint32_t out[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t v = 0;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) v |= gb[(4 * u + kk + rot) & 31] << (8 * kk);
      out[u] = v;
    }
    unsigned char* cb = reinterpret_cast<unsigned char*>(codes);
    *reinterpret_cast<uint4*>(cb + lut_byte(n, b, 0, NG)) = make_uint4(out[0], out[1], out[2], out[3]);
    *reinterpret_cast<uint4*>(cb + lut_byte(n, b, 16, NG)) = make_uint4(out[4], out[5], out[6], out[7]);
    scales[b * NG * 32 + n] = f64_to_f16_rne(s);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(codes + record_word(n, b, K, 8));
    dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
    dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
    scales[scale_index(n, b, scale_steps(K))] = f64_to_f16_rne(s);
  }
}

template <bool LUT>
__global__ void pack_int4_kernel(const float* __restrict__ w, int64_t N, int64_t K, uint32_t* __restrict__ codes,
                                 uint16_t* __restrict__ scales) {
  const int64_t nb = K / 128;
  const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= N * nb) return;
  const int64_t n = blk / nb, b = blk % nb;
  const float4* src = reinterpret_cast<const float4*>(w + n * K + b * 128);
  float mx = 0.f;
  for (int i = 0; i < 32; ++i) {
    const float4 v = src[i];
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  const double s = (double)mx / 7.0;
  uint32_t words[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) words[j] = 0u;
  for (int i = 0; i < 32; ++i) {
    const float4 v = src[i];
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int k = i * 4 + c;
      int q = 0;
      if (s != 0.0) {
        const double r = rint((double)vv[c] / s);
        q = r > 7.0 ? 7 : (r < -7.0 ? -7 : (int)r);
      }
      const int rr = k & 7;
      const int pos = (rr & 1) ? 14 + 2 * rr : 2 * rr;
      words[k >> 3] |= ((uint32_t)q & 0xFu) << pos;
    }
  }
  if constexpr (LUT) {
    // pair p (columns 2p, 2p + 1) as one byte, low nibble first; the two halves of
    // 32 bytes each rotated by n % 32
    uint32_t pb[64];
#pragma unroll
    for (int p = 0; p < 64; ++p) {
      uint32_t v = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = 2 * p + i, rr = k & 7;
        const int pos = (rr & 1) ? 14 + 2 * rr : 2 * rr;
        v |= ((words[k >> 3] >> pos) & 0xFu) << (4 * i);
      }
      pb[p] = v;
    }
    const int64_t NG = (N + 31) / 32;
    const int rot = (int)(n % 32);
    unsigned char* cb = reinterpret_cast<unsigned char*>(codes);
#pragma unroll
    for (int piece = 0; piece < 4; ++piece) {
      uint32_t out[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t v = 0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int t = 16 * piece + 4 * u + kk;
          v |= pb[32 * (t >> 5) + ((t & 31) + rot) % 32] << (8 * kk);
        }
        out[u] = v;
      }
      *reinterpret_cast<uint4*>(cb + lut4_byte(n, b, 16 * piece, NG)) = make_uint4(out[0], out[1], out[2], out[3]);
    }
    scales[b * NG * 32 + n] = f64_to_f16_rne(s);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(codes + record_word(n, b, K, 16));
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(words[4 * j], words[4 * j + 1], words[4 * j + 2], words[4 * j + 3]);
    scales[scale_index(n, b, scale_steps(K))] = f64_to_f16_rne(s);
  }
}

// One thread per (row, block): decodes the block's columns to int8 and copies
// its scale to row-major order.
__global__ void unpack_kernel(int format, const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                              int64_t N, int64_t K, int8_t* __restrict__ q, uint16_t* __restrict__ scales_out,
                              int* err) {
  const int64_t KB = K / 128;
  const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= N * KB) return;
  const int64_t n = blk / KB, b = blk % KB;
  int8_t* out = q + n * K + b * 128;
  bool bad = false;
  if (format == QMV_TERNARY2_LUT) {
    const int64_t NG = (N + 31) / 32;
    const unsigned char* cb = reinterpret_cast<const unsigned char*>(codes);
    for (int t = 0; t < 32; ++t) {
      const uint32_t v = cb[lut_byte(n, b, t, NG)];
      const int c = (int)((t + n) % 32);
      for (int i = 0; i < 4; ++i) {
        const uint32_t code = (v >> (2 * i)) & 3u;
        bad |= code == 3u;
        out[4 * c + i] = code == 1u ? 1 : (code == 2u ? -1 : 0);
      }
    }
    if (bad) atomicCAS(err, 0, QMV_ERR_CORRUPT);
    if (scales_out) scales_out[n * KB + b] = scales[b * NG * 32 + n];
    return;
  }
  if (format == QMV_INT4_LUT) {
    const int64_t NG = (N + 31) / 32;
    const unsigned char* cb = reinterpret_cast<const unsigned char*>(codes);
    for (int t = 0; t < 64; ++t) {
      const uint32_t v = cb[lut4_byte(n, b, t, NG)];
      const int p = 32 * (t >> 5) + (int)(((t & 31) + n) % 32);
      for (int i = 0; i < 2; ++i) {
        const int nib = (int)((v >> (4 * i)) & 0xFu);
        out[2 * p + i] = (int8_t)(nib >= 8 ? nib - 16 : nib);
      }
    }
    if (scales_out) scales_out[n * KB + b] = scales[b * NG * 32 + n];
    return;
  }
  const int bw = format == QMV_TERNARY2 ? 8 : 16;
  const uint32_t* src = codes + record_word(n, b, K, bw);
  for (int wi = 0; wi < bw; ++wi) {
    const uint32_t w = src[wi];
    if (format == QMV_TERNARY2) {
      for (int r = 0; r < 16; ++r) {
        const int pos = (r & 1) ? 15 + r : r;
        const uint32_t c = (w >> pos) & 3u;
        bad |= c == 3u;
        out[wi * 16 + r] = c == 1u ? 1 : (c == 2u ? -1 : 0);
      }
    } else {
      for (int r = 0; r < 8; ++r) {
        const int pos = (r & 1) ? 14 + 2 * r : 2 * r;
        const int v = (int)((w >> pos) & 0xFu);
        out[wi * 8 + r] = (int8_t)(v >= 8 ? v - 16 : v);
      }
    }
  }
  if (bad) atomicCAS(err, 0, QMV_ERR_CORRUPT);
  if (scales_out) scales_out[n * KB + b] = scales[scale_index(n, b, scale_steps(K))];
}

int pack_common(int format, const qmv_desc* desc, const float* w, void* packed, void* stream) {
  const bool lut = desc && ((format == QMV_TERNARY2 && desc->format == QMV_TERNARY2_LUT) ||
                            (format == QMV_INT4 && desc->format == QMV_INT4_LUT));
  int rc = lut ? check_lut_desc(desc) : check_desc(desc, format);
  if (rc) return rc;
  if (!w || !packed) return fail(QMV_ERR_ARG, "NULL w or packed");
  if (!aligned16(w) || !aligned16(packed)) return fail(QMV_ERR_ALIGN, "w and packed must be 16-byte aligned");
  char* base = static_cast<char*>(packed);
  uint32_t* codes = reinterpret_cast<uint32_t*>(base + desc->off[0]);
  uint16_t* scales = reinterpret_cast<uint16_t*>(base + desc->off[1]);
  const int64_t blocks = desc->N * (desc->K / 128);
  const int threads = 128;
  const int64_t grid = (blocks + threads - 1) / threads;
  if (grid > INT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "matrix too large for one pack launch");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // zero the padding rows of the last row group, the padding scales (rows past
  // N, blocks past K/128) and the alignment padding after each section, so
  // every byte is determined
  if (desc->N % (lut ? 32 : 16)) {
    cudaError_t e = cudaMemsetAsync(base + desc->off[0], 0, (size_t)desc->bytes[0], s);
    if (e != cudaSuccess) return cuda_fail(e, "zero padding rows");
  }
  if (desc->N % (lut ? 32 : 16) || (!lut && (desc->K / 128) % 8)) {
    cudaError_t e = cudaMemsetAsync(base + desc->off[1], 0, (size_t)desc->bytes[1], s);
    if (e != cudaSuccess) return cuda_fail(e, "zero padding scales");
  }
  const int64_t gaps[2][2] = {{desc->off[0] + desc->bytes[0], desc->off[1]},
                              {desc->off[1] + desc->bytes[1], desc->total_bytes}};
  for (const auto& gp : gaps) {
    if (gp[1] > gp[0]) {
      cudaError_t e = cudaMemsetAsync(base + gp[0], 0, (size_t)(gp[1] - gp[0]), s);
      if (e != cudaSuccess) return cuda_fail(e, "zero section padding");
    }
  }
  if (format == QMV_TERNARY2 && lut)
    pack_ternary_kernel<true><<<(unsigned)grid, threads, 0, s>>>(w, desc->N, desc->K, codes, scales);
  else if (format == QMV_TERNARY2)
    pack_ternary_kernel<false><<<(unsigned)grid, threads, 0, s>>>(w, desc->N, desc->K, codes, scales);
  else if (lut)
    pack_int4_kernel<true><<<(unsigned)grid, threads, 0, s>>>(w, desc->N, desc->K, codes, scales);
  else
    pack_int4_kernel<false><<<(unsigned)grid, threads, 0, s>>>(w, desc->N, desc->K, codes, scales);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  return QMV_OK;
}

}  // namespace
}  // namespace qmv

using namespace qmv;

extern "C" {

int qmv_pack_ternary(const qmv_desc* desc, const float* w, void* packed, void* stream) {
  return pack_common(QMV_TERNARY2, desc, w, packed, stream);
}

int qmv_pack_int4(const qmv_desc* desc, const float* w, void* packed, void* stream) {
  return pack_common(QMV_INT4, desc, w, packed, stream);
}

int qmv_unpack(const qmv_desc* desc, const void* packed, int8_t* q, uint16_t* scales, void* stream) {
  if (!desc) return fail(QMV_ERR_ARG, "desc is NULL");
  const int format = (int)desc->format;
  if (format != QMV_TERNARY2 && format != QMV_INT4 && format != QMV_TERNARY2_LUT && format != QMV_INT4_LUT)
    return fail(QMV_ERR_UNSUPPORTED, "qmv_unpack serves ternary and INT4 (either layout)");
  const bool lutf = format == QMV_TERNARY2_LUT || format == QMV_INT4_LUT;
  int rc = lutf ? check_lut_desc(desc) : check_desc(desc, format);
  if (rc) return rc;
  if (!packed || !q) return fail(QMV_ERR_ARG, "NULL packed or q");
  if (!aligned16(packed) || !aligned16(q) || (scales && !aligned16(scales)))
    return fail(QMV_ERR_ALIGN, "buffers must be 16-byte aligned");
  int* err = device_error_word();
  if (!err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  const char* base = static_cast<const char*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nblk = desc->N * (desc->K / 128);
  const int threads = 128;
  unpack_kernel<<<(unsigned)((nblk + threads - 1) / threads), threads, 0, s>>>(
      format, reinterpret_cast<const uint32_t*>(base + desc->off[0]),
      reinterpret_cast<const uint16_t*>(base + desc->off[1]), desc->N, desc->K, q, scales, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "unpack launch");
  return QMV_OK;
}

}  // extern "C"
