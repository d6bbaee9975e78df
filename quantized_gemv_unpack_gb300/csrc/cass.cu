// Cassandra lossless bf16 split ("Cassandra", sections 3.1-3.3) and its
// shared-exponent variant (Cassandra-2): the host-side offline transforms and
// the GPU draft / target paths.
//
// Offline (host): Wanda value pruning keeps the K/2 largest |w| * ||X[:,j]||_2
// of every row (bitmap), kept values keep sign + 3 high mantissa bits in the
// speculation data and 4 low mantissa bits in the verification data, their
// exponents are ranked by frequency over the whole tensor and written as unary
// codes (rank r = r zeros then a one), pruned values go to the verification
// data as raw bf16.
//
// GPU: one warp per row, rows strided over a persistent grid. A row keeps
// exactly K/2 values and prunes K/2, so lane l takes the kept values of rank
// k in [l*K2/32, (l+1)*K2/32) and the pruned values of the same ranks: every
// lane has the same work whatever the bitmap looks like, and no lane works
// per column. Each lane walks its ranks in order with bit cursors: over the
// exponent stream (the k-th one ends the k-th codeword; the zeros since the
// previous one are its rank), over the bitmap's ones (the column of the k-th
// kept value) and over its zeros (the column of the p-th pruned value). The
// cursors start from warp-wide selects: the row's words are scanned 128 at a
// time (four per lane, warp prefix sum of their bit counts) and each lane
// finds the word holding the one or zero of its first rank by a binary search
// over the lanes' prefix sums. Nibbles, sign bits and pruned halves are read
// in rank order from skewed shared-memory copies (one pad word per 8 or 32
// words, so that the 32 lanes' reads fall in distinct banks). Activations are
// staged per CTA as bf16 with all M rows of a column side by side (padded to
// 1, 2, 4 or 8), so one shared load gathers a column's activations; column j
// sits at unit j + (j >> sk), 2^sk being about the columns one lane covers,
// again to spread the lanes over the banks. Each product is exact in fp32
// (bf16 x bf16) and summed in fp32; the lanes' partial sums are reduced by
// shuffles. Every loop is bounded by the row's sizes; inconsistent streams set
// QMV_ERR_CORRUPT in the device error word.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "qmv_internal.cuh"

namespace qmv {
namespace {

// Warps per CTA: 32 where the kernel fits 64 registers a thread, else 16.
template <int MT, bool TARGET>
struct CassWarps {
  static constexpr int value = TARGET && MT > 5 ? 16 : 32;
};
inline int cass_warps(int M, bool target) { return target && M > 5 ? 16 : 32; }

__device__ __forceinline__ void flag(int* err) { atomicCAS(err, 0, (int)QMV_ERR_CORRUPT); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ----------------------------------------------------------------------------- rank walks

// Words of a skewed copy of n words with one pad word after every 2^SH.
__host__ __device__ constexpr size_t skewed_words(size_t n, int sh) { return n + (n >> sh) + 1; }
template <int SH>
__device__ __forceinline__ int skew(int w) { return w + (w >> SH); }

// Activation staging: unit j + (j >> sk) holds the M rows of column j, as
// P bf16 (one fp32 when M = 1, which saves the widening in the walk).
template <int MT>
struct XPad {
  static constexpr int P = MT == 1 ? 1 : MT == 2 ? 2 : MT <= 4 ? 4 : 8;
};
__host__ __device__ inline size_t xs_bytes(size_t K, int sk, int P) {
  return ((K + (K >> sk) + 1) * (size_t)(P == 1 ? 4 : P * 2) + 15) / 16 * 16;
}

template <int MT>
__device__ void stage_x(uint16_t* xs, const uint16_t* x, int ldx, int K, int sk) {
  constexpr int P = XPad<MT>::P;
  if constexpr (P == 1) {
    float* xf = reinterpret_cast<float*>(xs);
    for (int j = threadIdx.x; j < K; j += blockDim.x) xf[j + (j >> sk)] = __uint_as_float((uint32_t)x[j] << 16);
  } else {
    for (int i = threadIdx.x; i < K * P; i += blockDim.x) {
      const int j = i / P, m = i % P;
      xs[(size_t)(j + (j >> sk)) * P + m] = m < MT ? x[(size_t)m * ldx + j] : (uint16_t)0;
    }
  }
}

template <int MT>
__device__ __forceinline__ void x_gather(const uint16_t* xs, int j, int sk, float (&xv)[MT]) {
  constexpr int P = XPad<MT>::P;
  const int u = j + (j >> sk);
  uint32_t w[P == 1 ? 1 : P / 2];
  if constexpr (P == 1) {
    xv[0] = reinterpret_cast<const float*>(xs)[u];
    return;
  } else if constexpr (P == 2) {
    w[0] = reinterpret_cast<const uint32_t*>(xs)[u];
  } else if constexpr (P == 4) {
    const uint2 v = reinterpret_cast<const uint2*>(xs)[u];
    w[0] = v.x, w[1] = v.y;
  } else {
    const uint4 v = reinterpret_cast<const uint4*>(xs)[u];
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  }
  if constexpr (P > 1) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
      xv[m] = __uint_as_float(m & 1 ? w[m >> 1] & 0xffff0000u : w[m >> 1] << 16);
  }
}

// Copies n words to dst[skew<SH>(w)]; 16-byte loads when the source allows.
template <int SH>
__device__ __forceinline__ void stage_words(uint32_t* dst, const uint32_t* src, int n) {
  const int lane = threadIdx.x & 31;
  if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int i = lane; i < n / 4; i += 32) {
      const uint4 v = __ldg(s4 + i);
      uint32_t* d = dst + skew<SH>(4 * i);  // 4 words never straddle a pad (SH >= 2)
      d[0] = v.x, d[1] = v.y, d[2] = v.z, d[3] = v.w;
    }
  } else {
    for (int w = lane; w < n; w += 32) dst[skew<SH>(w)] = __ldg(src + w);
  }
}

// Position (0..31) of the r-th set bit of x (r < popc(x)).
__device__ __forceinline__ int select_in_word(uint32_t x, int r) {
  int p = 0, c;
  c = __popc(x & 0xFFFFu);
  if (r >= c) r -= c, x >>= 16, p += 16;
  c = __popc(x & 0xFFu);
  if (r >= c) r -= c, x >>= 8, p += 8;
  c = __popc(x & 0xFu);
  if (r >= c) r -= c, x >>= 4, p += 4;
  c = __popc(x & 0x3u);
  if (r >= c) r -= c, x >>= 2, p += 2;
  if (r >= (int)(x & 1u)) p += 1;
  return p;
}

struct Hit {
  uint32_t w;  // the word holding the target bit
  int r;       // the target's rank among the word's set bits
  int wi;      // the word's index (past the end: not found)
};
__device__ __forceinline__ int hit_pos(const Hit& h) { return h.wi * 32 + select_in_word(h.w, h.r); }

// One warp-collective step of a select: q holds words c + 4*lane + 0..3 of an
// array (0 past its end) and `carry` counts the set bits before word c. If the
// lane's target rank t falls in these 128 words, h records where. Returns the
// set bits in the 128 words.
__device__ __forceinline__ int select_chunk(const uint32_t (&q)[4], int c, int t, int carry, Hit& h) {
  const int lane = threadIdx.x & 31;
  const int v = __popc(q[0]) + __popc(q[1]) + __popc(q[2]) + __popc(q[3]);
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  const int excl = incl - v;
  const int tot = __shfl_sync(0xffffffffu, incl, 31);
  const int tt = t - carry;
  int j = 0;  // the last lane whose words start at or before rank tt
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const int e = __shfl_sync(0xffffffffu, excl, j + s);
    if (e <= tt) j += s;
  }
  const int ej = __shfl_sync(0xffffffffu, excl, j);
  const uint32_t a0 = __shfl_sync(0xffffffffu, q[0], j), a1 = __shfl_sync(0xffffffffu, q[1], j);
  const uint32_t a2 = __shfl_sync(0xffffffffu, q[2], j), a3 = __shfl_sync(0xffffffffu, q[3], j);
  if (tt >= 0 && tt < tot) {
    int r = tt - ej, sel = 0;
    uint32_t x = a0;
    if (r >= __popc(a0)) {
      r -= __popc(a0), x = a1, sel = 1;
      if (r >= __popc(a1)) {
        r -= __popc(a1), x = a2, sel = 2;
        if (r >= __popc(a2)) r -= __popc(a2), x = a3, sel = 3;
      }
    }
    h.w = x, h.r = r, h.wi = c + 4 * j + sel;
  }
  return tot;
}

// Loads words c + 4*lane + 0..3 of a row (0 past n), 16 bytes at a time when aligned.
__device__ __forceinline__ void load_quad(const uint32_t* src, int n, int c, bool vec, uint32_t (&q)[4]) {
  const int w0 = c + 4 * (threadIdx.x & 31);
  if (vec) {
    const uint4 v = w0 < n ? __ldg(reinterpret_cast<const uint4*>(src + w0)) : make_uint4(0, 0, 0, 0);
    q[0] = v.x, q[1] = v.y, q[2] = v.z, q[3] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = w0 + i < n ? __ldg(src + w0 + i) : 0u;
  }
}

// Stages a row's bitmap (KW words) and finds the column of the lane's first
// kept value (rank k0 among the ones) and first pruned value (rank k0 among
// the zeros). Returns the number of ones; `clean` (warp-uniform) says that no
// word is all zeros or all ones, so the cursors never skip a whole word.
__device__ __forceinline__ int bitmap_selects(const uint32_t* src, uint32_t* bm_s, int KW, int k0, Hit& h1, Hit& h0,
                                              bool& clean) {
  const bool vec = (KW & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  int ones = 0, zeros = 0;
  h1.wi = h0.wi = KW;
  h1.w = h0.w = 0u;
  h1.r = h0.r = 0;
  bool flat = false;
  for (int c = 0; c < KW; c += 128) {
    uint32_t q[4], z[4];
    load_quad(src, KW, c, vec, q);
    const int w0 = c + 4 * (threadIdx.x & 31);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (w0 + i < KW) {
        bm_s[w0 + i] = q[i];
        flat |= q[i] == 0u || q[i] == 0xffffffffu;
      }
      z[i] = w0 + i < KW ? ~q[i] : 0u;
    }
    ones += select_chunk(q, c, k0, ones, h1);
    zeros += select_chunk(z, c, k0, zeros, h0);
  }
  clean = !__any_sync(0xffffffffu, flat);
  return ones;
}

// A forward cursor over the set bits (INV: the clear bits) of a word array,
// with the next word preloaded.
struct Cursor {
  uint32_t w;   // the unread bits of word wi (inverted for INV)
  uint32_t nx;  // word wi + 1 as stored
  int wi;
};

template <bool INV>
__device__ __forceinline__ uint32_t cursor_raw(const uint32_t* s, int nw, int i) {
  return i < nw ? s[i] : (INV ? 0xffffffffu : 0u);
}

template <bool INV>
__device__ __forceinline__ Cursor cursor_at(const uint32_t* s, int nw, int pos) {
  Cursor c;
  c.wi = pos >> 5;
  const uint32_t raw = cursor_raw<INV>(s, nw, c.wi);
  c.w = (INV ? ~raw : raw) & (0xffffffffu << (pos & 31));
  c.nx = cursor_raw<INV>(s, nw, c.wi + 1);
  return c;
}

// The next bit at or after the cursor (its position); the cursor moves past
// it. Without SAFE the caller guarantees that no word before the last bit it
// asks for is empty, so one step to the preloaded word always finds a bit.
// With SAFE empty words are skipped, and running off the end sets `bad`.
template <bool INV, bool SAFE>
__device__ __forceinline__ int cursor_next(Cursor& c, const uint32_t* s, int nw, bool& bad) {
  if (c.w == 0) {
    c.w = INV ? ~c.nx : c.nx;
    ++c.wi;
    c.nx = cursor_raw<INV>(s, nw, c.wi + 1);
  }
  if (SAFE) {
    while (c.w == 0) {
      if (c.wi >= nw) {
        bad = true;
        return 0;
      }
      c.w = INV ? ~c.nx : c.nx;
      ++c.wi;
      c.nx = cursor_raw<INV>(s, nw, c.wi + 1);
    }
  }
  const int b = __ffs(c.w) - 1;
  c.w &= c.w - 1;
  return c.wi * 32 + b;
}

// The fast-walk step over a shared-memory array (`base` its shared address):
// the caller guarantees that the bit exists and that no word before it is
// empty, and pads the array so that word wi + 1 can be read. The refill is
// branch-free and only the lanes that refill load (a predicated load), which
// keeps the cursors off the shared-memory banks most steps.
template <bool INV>
__device__ __forceinline__ int cursor_step(Cursor& c, uint32_t base) {
  const uint32_t e = c.w == 0;
  c.w = e ? (INV ? ~c.nx : c.nx) : c.w;
  c.wi += e;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p ld.shared.u32 %0, [%2];\n\t}"
      : "+r"(c.nx)
      : "r"(e), "r"(base + 4u * (uint32_t)(c.wi + 1)));
  const int b = __ffs(c.w) - 1;
  c.w &= c.w - 1;
  return c.wi * 32 + b;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

template <int MT>
__device__ __forceinline__ void accumulate(const uint16_t* xs, int j, int sk, float w, float (&acc)[MT]) {
  float xv[MT];
  x_gather<MT>(xs, j, sk, xv);
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = fmaf(w, xv[m], acc[m]);
}

template <int MT>
__device__ __forceinline__ void store_row(float (&acc)[MT], float* y, int ldy, int n) {
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) y[(size_t)m * ldy + n] = v;
  }
}

// ----------------------------------------------------------------------------- Cassandra-1

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
  uint16_t* w_out;           // [N][K] or null (written by the WOUT kernels only)
  int64_t stream_words;
  int N, K, ldx, ldy, n_symbols;
  int sk;                    // activation unit skew shift
  int scap;                  // stream words a warp stages (longer rows are read in place)
  int* err;
};

// Shared memory of one warp: bitmap, nibbles (+ target: low nibbles), staged
// stream; the bitmap and the stream carry two pad words for the fast walk's
// read-ahead. Pruned halves are read from global memory, each lane's run
// being contiguous.
__host__ __device__ inline size_t cass_per_warp(size_t K, size_t scap, bool target) {
  const size_t w = K / 32 + 2 + skewed_words(K / 16, 3) + (target ? skewed_words(K / 16, 3) : 0) + scap + 2;
  return (w * 4 + 15) / 16 * 16;
}

// Bytes of the (rank, nibble) -> draft value table: the fp32 bits of the bf16
// draft value S<<15 | E<<7 | m_hi<<4 (shifted left by 16) for every codebook rank
// and sign/high-mantissa nibble; the target ORs the low mantissa nibble in at
// bits 16..19.
__host__ __device__ inline size_t cass_tab_bytes(int n_symbols) { return (size_t)n_symbols * 64; }

// The staged row one lane walks.
struct CassRow {
  const uint32_t *bm, *sm, *lo, *st;
  const uint16_t* prg;  // the row's pruned halves (global)
  const uint32_t* tab;
  const uint16_t* xs;
  uint16_t* wrow;
  int KW, nsw, nsym, sk;
  int k0, cnt;
  int send;            // where codeword k0 starts in the stream
  int kpos, zpos;      // columns of kept value k0 and pruned value k0
};

// Kept value k and pruned value k for k in [k0, k0 + cnt): see the file comment.
template <int MT, bool TARGET, bool WOUT, bool SAFE>
__device__ __forceinline__ void cass_walk(const CassRow& r, float (&acc)[MT], bool& bad) {
  Cursor cs = cursor_at<false>(r.st, r.nsw, r.send);
  Cursor ck = cursor_at<false>(r.bm, r.KW, r.kpos);
  Cursor cz = cursor_at<true>(r.bm, r.KW, r.zpos);
  int send = r.send;
  uint32_t smw = r.sm[skew<3>(r.k0 >> 3)];
  uint32_t low = TARGET ? r.lo[skew<3>(r.k0 >> 3)] : 0u;
  for (int k = r.k0; k < r.k0 + r.cnt; ++k) {
    const int sp = cursor_next<false, SAFE>(cs, r.st, r.nsw, bad);
    int rank = sp - send;
    send = sp + 1;
    if ((unsigned)rank >= (unsigned)r.nsym) bad = true, rank = 0;
    const int j = cursor_next<false, SAFE>(ck, r.bm, r.KW, bad);
    if ((k & 7) == 0) {
      smw = r.sm[skew<3>(k >> 3)];
      if (TARGET) low = r.lo[skew<3>(k >> 3)];
    }
    const int sh = (k & 7) * 4;
    uint32_t v = r.tab[rank * 16 + ((smw >> sh) & 0xFu)];
    if (TARGET) v |= ((low >> sh) & 0xFu) << 16;
    if (WOUT) r.wrow[j] = (uint16_t)(v >> 16);
    accumulate<MT>(r.xs, j, r.sk, __uint_as_float(v), acc);
    if (TARGET || WOUT) {
      const int jz = cursor_next<true, SAFE>(cz, r.bm, r.KW, bad);
      uint32_t pv = 0;
      if (TARGET) {
        pv = __ldg(r.prg + k);
        accumulate<MT>(r.xs, jz, r.sk, __uint_as_float(pv << 16), acc);
      }
      if (WOUT) r.wrow[jz] = (uint16_t)pv;
    }
  }
}

// Pruned halves of ranks k .. k + 7 (16-byte aligned: k is a multiple of 8).
__device__ __forceinline__ uint4 pruned_block(const uint16_t* prg, int k) {
  return __ldg(reinterpret_cast<const uint4*>(prg + k));
}
__device__ __forceinline__ uint32_t block_half(const uint4& v, int u) {
  const uint32_t w = u < 2 ? v.x : u < 4 ? v.y : u < 6 ? v.z : v.w;
  return u & 1 ? w >> 16 : w & 0xFFFFu;
}

// The same walk for rows with no empty word in the way and K a multiple of
// 512 (every lane's ranks start at a multiple of 8 and come in blocks of 8):
// unrolled by 8, nibble shifts constant, cursors branch-free.
template <int MT, bool TARGET>
__device__ __forceinline__ void cass_walk8(const CassRow& r, float (&acc)[MT], bool& bad) {
  Cursor cs = cursor_at<false>(r.st, r.nsw, r.send);
  Cursor ck = cursor_at<false>(r.bm, r.KW, r.kpos);
  Cursor cz = cursor_at<true>(r.bm, r.KW, r.zpos);
  const uint32_t st_base = smem_u32(r.st), bm_base = smem_u32(r.bm);
  int send = r.send;
  // ranks are clamped to the codebook for the lookup and their maximum checked once
  unsigned rmax = 0;
  const unsigned rlast = (unsigned)r.nsym - 1u;
  uint4 pnext = TARGET ? pruned_block(r.prg, r.k0) : make_uint4(0, 0, 0, 0);
  for (int k = r.k0; k < r.k0 + r.cnt; k += 8) {
    const uint32_t smw = r.sm[skew<3>(k >> 3)];
    const uint32_t low = TARGET ? r.lo[skew<3>(k >> 3)] : 0u;
    const uint4 pcur = pnext;
    if (TARGET && k + 8 < r.k0 + r.cnt) pnext = pruned_block(r.prg, k + 8);  // one block ahead
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sp = cursor_step<false>(cs, st_base);
      const unsigned rank = (unsigned)(sp - send);
      send = sp + 1;
      rmax = max(rmax, rank);
      uint32_t v = r.tab[min(rank, rlast) * 16 + ((smw >> (4 * u)) & 0xFu)];
      if (TARGET) v |= ((low >> (4 * u)) & 0xFu) << 16;
      accumulate<MT>(r.xs, cursor_step<false>(ck, bm_base), r.sk, __uint_as_float(v), acc);
      if (TARGET)
        accumulate<MT>(r.xs, cursor_step<true>(cz, bm_base), r.sk, __uint_as_float(block_half(pcur, u) << 16), acc);
    }
  }
  if (rmax > rlast) bad = true;
}

template <int MT, bool TARGET, bool WOUT>
__global__ void __launch_bounds__(CassWarps<MT, TARGET>::value * 32) cass_kernel(const CassArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int P = XPad<MT>::P;
  const int K = a.K, K2 = K / 2, KW = K / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  const size_t xb = xs_bytes(K, a.sk, P);
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + xb);
  uint32_t* bm_s = reinterpret_cast<uint32_t*>(smem + xb + cass_tab_bytes(a.n_symbols) +
                                               (size_t)warp * cass_per_warp(K, a.scap, TARGET));
  uint32_t* sm_s = bm_s + KW + 2;
  uint32_t* lo_s = sm_s + skewed_words(K / 16, 3);
  uint32_t* st_s = lo_s + (TARGET ? skewed_words(K / 16, 3) : 0);

  for (int i = threadIdx.x; i < a.n_symbols * 16; i += blockDim.x) {
    const uint32_t nib = i & 15;
    tab[i] = (((nib & 8u) << 12) | ((uint32_t)a.codebook[i >> 4] << 7) | ((nib & 7u) << 4)) << 16;
  }
  stage_x<MT>(xs, a.x, a.ldx, K, a.sk);
  __syncthreads();

  CassRow r;
  r.bm = bm_s, r.sm = sm_s, r.lo = lo_s, r.tab = tab, r.xs = xs;
  r.KW = KW, r.nsym = a.n_symbols, r.sk = a.sk;
  r.k0 = (int)(((int64_t)lane * K2) >> 5);
  r.cnt = (int)(((int64_t)(lane + 1) * K2) >> 5) - r.k0;
  for (int n = blockIdx.x * nwarps + warp; n < a.N; n += gridDim.x * nwarps) {
    // ---- stage the row: nibbles (skewed), bitmap with the two selects, stream with one
    stage_words<3>(sm_s, a.signmant + (size_t)n * (K / 16), K / 16);
    if (TARGET) stage_words<3>(lo_s, a.mlo + (size_t)n * (K / 16), K / 16);
    r.prg = a.pruned + (size_t)n * K2;
    Hit h1, h0;
    bool clean;
    const int ones = bitmap_selects(a.bitmap + (size_t)n * KW, bm_s, KW, r.k0, h1, h0, clean);
    uint32_t s0 = __ldg(a.rowstart + n), s1 = __ldg(a.rowstart + n + 1);
    bool bad = ones != K2;
    if (s1 < s0 || (int64_t)s1 > a.stream_words) bad = true, s1 = s0;
    const int nsw = (int)(s1 - s0);
    const uint32_t* sg = a.stream + s0;
    const bool fits = nsw <= a.scap;
    Hit hs;
    hs.w = 0u, hs.r = 0, hs.wi = nsw;
    int codes = 0;
    int first_zero = nsw, last_set = -1;  // an empty word before the last one needs the safe walk
    for (int c = 0; c < nsw; c += 128) {
      uint32_t q[4];
      load_quad(sg, nsw, c, false, q);
      const int w0 = c + 4 * lane;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (w0 + i < nsw) {
          if (fits) st_s[w0 + i] = q[i];
          if (q[i]) last_set = w0 + i;
          else first_zero = min(first_zero, w0 + i);
        }
      }
      codes += select_chunk(q, c, r.k0 - 1, codes, hs);
    }
    first_zero = __reduce_min_sync(0xffffffffu, first_zero);
    last_set = __reduce_max_sync(0xffffffffu, last_set);
    if (codes != K2) bad = true;
    __syncwarp();

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    bool lbad = false;
    if (!bad && r.cnt > 0) {
      r.nsw = nsw;
      r.send = r.k0 == 0 ? 0 : hit_pos(hs) + 1;
      r.kpos = hit_pos(h1);
      r.zpos = hit_pos(h0);
      r.wrow = WOUT ? a.w_out + (size_t)n * K : nullptr;
      if (!WOUT && (K & 511) == 0 && fits && clean && first_zero > last_set) {
        r.st = st_s;
        cass_walk8<MT, TARGET>(r, acc, lbad);
      } else if (fits && clean && first_zero > last_set) {
        r.st = st_s;
        cass_walk<MT, TARGET, WOUT, false>(r, acc, lbad);
      } else {
        r.st = fits ? st_s : sg;
        cass_walk<MT, TARGET, WOUT, true>(r, acc, lbad);
      }
    }
    if ((__any_sync(0xffffffffu, lbad) || bad) && lane == 0) flag(a.err);
    if (a.y) store_row<MT>(acc, a.y, a.ldy, n);
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
  uint16_t* w_out;           // [N][K] or null (written by the WOUT kernels only)
  int N, K, ldx, ldy;
  int sk;                    // activation unit skew shift
  int* err;
};

__host__ __device__ inline size_t cassmx_per_warp(size_t K, bool target) {
  // bitmap, signs, draft nibbles, group scales (+ target: low nibbles); pruned halves stay in global memory
  const size_t w = K / 32 + 2 + K / 64 + skewed_words(K / 16, 3) + K / 64 + (target ? skewed_words(K / 16, 3) : 0);
  return (w * 4 + 15) / 16 * 16;
}

struct MxRow {
  const uint32_t *bm, *sg, *dn, *ln;
  const uint16_t* prg;  // the row's pruned halves (global)
  const float* sc;
  const uint16_t* xs;
  uint16_t* wrow;
  int KW, sk, k0, cnt, kpos, zpos;
};

// The rank walk with no exponent stream: the kept value of rank k is its
// nibble(s) times the fp32 scale of its group of 32 (2^(g - 134) for the
// target, 2^(g - 130) for the draft), sign from the sign bits; exact in fp32
// and in bf16.
template <int MT, bool TARGET, bool WOUT, bool SAFE>
__device__ __forceinline__ void cassmx_walk(const MxRow& r, float (&acc)[MT], bool& bad) {
  Cursor ck = cursor_at<false>(r.bm, r.KW, r.kpos);
  Cursor cz = cursor_at<true>(r.bm, r.KW, r.zpos);
  uint32_t dw = r.dn[skew<3>(r.k0 >> 3)];
  uint32_t lw = TARGET ? r.ln[skew<3>(r.k0 >> 3)] : 0u;
  uint32_t sgw = r.sg[r.k0 >> 5];
  float scl = r.sc[r.k0 >> 5];
  for (int k = r.k0; k < r.k0 + r.cnt; ++k) {
    const int j = cursor_next<false, SAFE>(ck, r.bm, r.KW, bad);
    if ((k & 7) == 0) {
      dw = r.dn[skew<3>(k >> 3)];
      if (TARGET) lw = r.ln[skew<3>(k >> 3)];
    }
    if ((k & 31) == 0) sgw = r.sg[k >> 5], scl = r.sc[k >> 5];
    const int sh = (k & 7) * 4;
    uint32_t mag = (dw >> sh) & 0xFu;
    if (TARGET) mag = (mag << 4) | ((lw >> sh) & 0xFu);
    float v = (float)mag * scl;
    if ((sgw >> (k & 31)) & 1u) v = -v;
    if (WOUT) r.wrow[j] = (uint16_t)(__float_as_uint(v) >> 16);
    accumulate<MT>(r.xs, j, r.sk, v, acc);
    if (TARGET || WOUT) {
      const int jz = cursor_next<true, SAFE>(cz, r.bm, r.KW, bad);
      uint32_t pv = 0;
      if (TARGET) {
        pv = __ldg(r.prg + k);
        accumulate<MT>(r.xs, jz, r.sk, __uint_as_float(pv << 16), acc);
      }
      if (WOUT) r.wrow[jz] = (uint16_t)pv;
    }
  }
}

// Unrolled by 8 for clean rows and K a multiple of 512, as cass_walk8.
template <int MT, bool TARGET>
__device__ __forceinline__ void cassmx_walk8(const MxRow& r, float (&acc)[MT]) {
  Cursor ck = cursor_at<false>(r.bm, r.KW, r.kpos);
  Cursor cz = cursor_at<true>(r.bm, r.KW, r.zpos);
  const uint32_t bm_base = smem_u32(r.bm);
  uint4 pnext = TARGET ? pruned_block(r.prg, r.k0) : make_uint4(0, 0, 0, 0);
  for (int k = r.k0; k < r.k0 + r.cnt; k += 8) {
    const uint32_t dw = r.dn[skew<3>(k >> 3)];
    const uint32_t lw = TARGET ? r.ln[skew<3>(k >> 3)] : 0u;
    const uint32_t sgb = r.sg[k >> 5] >> (k & 24);
    const float scl = r.sc[k >> 5];
    const uint4 pcur = pnext;
    if (TARGET && k + 8 < r.k0 + r.cnt) pnext = pruned_block(r.prg, k + 8);  // one block ahead
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t mag = (dw >> (4 * u)) & 0xFu;
      if (TARGET) mag = (mag << 4) | ((lw >> (4 * u)) & 0xFu);
      const float v = __uint_as_float(__float_as_uint((float)mag * scl) ^ (((sgb >> u) & 1u) << 31));
      accumulate<MT>(r.xs, cursor_step<false>(ck, bm_base), r.sk, v, acc);
      if (TARGET)
        accumulate<MT>(r.xs, cursor_step<true>(cz, bm_base), r.sk, __uint_as_float(block_half(pcur, u) << 16), acc);
    }
  }
}

template <int MT, bool TARGET, bool WOUT>
__global__ void __launch_bounds__(CassWarps<MT, TARGET>::value * 32) cassmx_kernel(const CassMxArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int P = XPad<MT>::P;
  const int K = a.K, K2 = K / 2, KW = K / 32, KG = K / 64;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  const size_t xb = xs_bytes(K, a.sk, P);
  uint32_t* bm_s = reinterpret_cast<uint32_t*>(smem + xb + (size_t)warp * cassmx_per_warp(K, TARGET));
  uint32_t* sg_s = bm_s + KW + 2;
  uint32_t* dn_s = sg_s + KG;
  float* sc_s = reinterpret_cast<float*>(dn_s + skewed_words(K / 16, 3));
  uint32_t* ln_s = reinterpret_cast<uint32_t*>(sc_s + KG);

  stage_x<MT>(xs, a.x, a.ldx, K, a.sk);
  __syncthreads();

  MxRow r;
  r.bm = bm_s, r.sg = sg_s, r.dn = dn_s, r.ln = ln_s, r.sc = sc_s, r.xs = xs;
  r.KW = KW, r.sk = a.sk;
  r.k0 = (int)(((int64_t)lane * K2) >> 5);
  r.cnt = (int)(((int64_t)(lane + 1) * K2) >> 5) - r.k0;
  for (int n = blockIdx.x * nwarps + warp; n < a.N; n += gridDim.x * nwarps) {
    for (int i = lane; i < KG; i += 32) {
      sg_s[i] = __ldg(a.signs + (size_t)n * KG + i);
      sc_s[i] = ldexpf(1.f, (int)__ldg(a.gexp + (size_t)n * KG + i) - (TARGET ? 134 : 130));
    }
    stage_words<3>(dn_s, a.dnib + (size_t)n * (K / 16), K / 16);
    if (TARGET) stage_words<3>(ln_s, a.lnib + (size_t)n * (K / 16), K / 16);
    r.prg = a.pruned + (size_t)n * K2;
    Hit h1, h0;
    bool clean;
    const bool bad = bitmap_selects(a.bitmap + (size_t)n * KW, bm_s, KW, r.k0, h1, h0, clean) != K2;
    __syncwarp();

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    bool lbad = false;
    if (!bad && r.cnt > 0) {
      r.kpos = hit_pos(h1);
      r.zpos = hit_pos(h0);
      r.wrow = WOUT ? a.w_out + (size_t)n * K : nullptr;
      if (!WOUT && (K & 511) == 0 && clean) cassmx_walk8<MT, TARGET>(r, acc);
      else if (clean) cassmx_walk<MT, TARGET, WOUT, false>(r, acc, lbad);
      else cassmx_walk<MT, TARGET, WOUT, true>(r, acc, lbad);
    }
    if ((__any_sync(0xffffffffu, lbad) || bad) && lane == 0) flag(a.err);
    if (a.y) store_row<MT>(acc, a.y, a.ldy, n);
    __syncwarp();  // the staged row buffers are reused by the next row
  }
}

// Activation unit skew: 2^sk about the K/32 columns one lane covers.
inline int x_skew(int K) {
  int sk = 0;
  while ((2 << sk) <= K / 32) ++sk;
  return sk;
}

template <class Args>
int launch_rows(const void* kern, const Args& a, int max_warps, size_t fixed, size_t per_warp, const char* what,
                cudaStream_t s) {
  const size_t cap = 227 * 1024 - 1024;
  if (fixed + per_warp > cap) return fail(QMV_ERR_UNSUPPORTED, "K=%d does not fit shared memory", a.K);
  const int warps = (int)std::min<size_t>(max_warps, (cap - fixed) / per_warp);
  const size_t smem = fixed + per_warp * warps;
  int per_sm = 0;
  int rc = kernel_fit(kern, warps * 32, smem, &per_sm);
  if (rc) return rc;
  const int grid = std::max(1, std::min(sm_count() * per_sm, (a.N + warps - 1) / warps));
  void* args[] = {const_cast<Args*>(&a)};
  cudaError_t e = cudaLaunchKernel(kern, grid, warps * 32, args, smem, s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return QMV_OK;
}

// Kernels with M = 1..8 activation rows; a dense w_out is written by the
// M = 1 WOUT variant (which then also serves y when M = 1), so the matvec
// kernels carry no per-value stores.
template <template <int, bool, bool> class Pick, class Args, bool TARGET>
int launch_pair(Args& a, int M, size_t fixed_extra, size_t per_warp, const char* what, cudaStream_t s) {
  if (M < 1 || M > 8) return fail(QMV_ERR_ARG, "M=%d outside 1..8", M);
  const int P = M == 1 ? 1 : M == 2 ? 2 : M <= 4 ? 4 : 8;
  int rc = QMV_OK;
  if (a.w_out) {
    Args b = a;
    if (M != 1) b.y = nullptr;
    rc = launch_rows(Pick<1, TARGET, true>::get(), b, cass_warps(1, TARGET), xs_bytes(a.K, a.sk, 1) + fixed_extra,
                     per_warp, what, s);
    if (rc || M == 1 || !a.y) return rc;
  }
  if (!a.y) return rc;
  Args b = a;
  b.w_out = nullptr;
  const void* kern = nullptr;
  switch (M) {
    case 1: kern = Pick<1, TARGET, false>::get(); break;
    case 2: kern = Pick<2, TARGET, false>::get(); break;
    case 3: kern = Pick<3, TARGET, false>::get(); break;
    case 4: kern = Pick<4, TARGET, false>::get(); break;
    case 5: kern = Pick<5, TARGET, false>::get(); break;
    case 6: kern = Pick<6, TARGET, false>::get(); break;
    case 7: kern = Pick<7, TARGET, false>::get(); break;
    default: kern = Pick<8, TARGET, false>::get(); break;
  }
  return launch_rows(kern, b, cass_warps(M, TARGET), xs_bytes(a.K, a.sk, P) + fixed_extra, per_warp, what, s);
}

template <int MT, bool TARGET, bool WOUT>
struct PickCass {
  static const void* get() { return (const void*)cass_kernel<MT, TARGET, WOUT>; }
};
template <int MT, bool TARGET, bool WOUT>
struct PickCassMx {
  static const void* get() { return (const void*)cassmx_kernel<MT, TARGET, WOUT>; }
};

template <bool TARGET>
int launch_cassmx(CassMxArgs& a, int M, cudaStream_t s) {
  a.sk = x_skew(a.K);
  return launch_pair<PickCassMx, CassMxArgs, TARGET>(a, M, 0, cassmx_per_warp(a.K, TARGET), "cassandra-2 launch", s);
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
int launch_cass(CassArgs& a, int M, cudaStream_t s) {
  a.sk = x_skew(a.K);
  a.scap = std::max(4, a.K / 8);  // 4 bits per kept value; longer rows are read in place
  return launch_pair<PickCass, CassArgs, TARGET>(a, M, cass_tab_bytes(a.n_symbols), cass_per_warp(a.K, a.scap, TARGET),
                                                "cassandra launch", s);
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

// Argument checks shared by the draft, target and draft-then-verify calls.
int check_cass_call(const qmv_desc* d, const void* packed, const void* x, int M, int64_t ldx, const float* y,
                    int64_t ldy, const uint16_t* w_out) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  const bool mx = d->abi_version == QMV_ABI_VERSION && d->format == QMV_CASS_MX;
  int rc = mx ? check_cassmx_desc(d) : check_cass_desc(d);
  if (rc) return rc;
  if (M < 1 || M > 8) return fail(QMV_ERR_ARG, "M=%d outside 1..8", M);
  if (!packed || !x) return fail(QMV_ERR_ARG, "NULL packed or x");
  if (!aligned16(packed) || !aligned16(x) || (y && !aligned16(y)) || (w_out && !aligned16(w_out)))
    return fail(QMV_ERR_ALIGN, "buffers must be 16-byte aligned");
  if (ldx < d->K || (y && ldy < d->N)) return fail(QMV_ERR_ARG, "ldx < K or ldy < N");
  if (ldx % 8) return fail(QMV_ERR_ALIGN, "ldx=%lld must be a multiple of 8 (16-byte rows)", (long long)ldx);
  if (ldx > INT32_MAX || ldy > INT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "leading dimension too large");
  return QMV_OK;
}

int run_cass(bool target, const qmv_desc* d, const void* packed, const void* x, int M, int64_t ldx, float* y,
             int64_t ldy, uint16_t* w_out, void* stream) {
  int rc = check_cass_call(d, packed, x, M, ldx, y, ldy, w_out);
  if (rc) return rc;
  const bool mx = d->format == QMV_CASS_MX;
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

int cass_speculate_step(const qmv_desc* desc, const void* packed, const void* x_bf16, int n_draft, int64_t ldx,
                        float* y_draft, float* y_target, int64_t ldy, void* stream) {
  if (n_draft < 1 || n_draft > 7) return fail(QMV_ERR_ARG, "n_draft=%d outside 1..7", n_draft);
  if (!y_draft || !y_target) return fail(QMV_ERR_ARG, "NULL y_draft or y_target");
  // all arguments are checked before the first launch
  int rc = check_cass_call(desc, packed, x_bf16, n_draft + 1, ldx, y_target, ldy, nullptr);
  if (rc) return rc;
  if (!aligned16(y_draft)) return fail(QMV_ERR_ALIGN, "y_draft must be 16-byte aligned");
  if (y_draft + (size_t)(n_draft - 1) * ldy + desc->N > y_target && y_target + (size_t)n_draft * ldy + desc->N > y_draft)
    return fail(QMV_ERR_ARG, "y_draft and y_target overlap");
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  // the draft tokens in order: draft token d is produced from activation row d
  for (int d = 0; d < n_draft; ++d) {
    rc = run_cass(false, desc, packed, x + (size_t)d * ldx, 1, ldx, y_draft + (size_t)d * ldy, ldy, nullptr, stream);
    if (rc) return rc;
  }
  // one target pass verifies the current token and all draft tokens
  return run_cass(true, desc, packed, x, n_draft + 1, ldx, y_target, ldy, nullptr, stream);
}

}  // extern "C"
