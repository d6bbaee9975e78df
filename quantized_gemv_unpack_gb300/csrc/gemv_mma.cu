// Fused dequantize-and-matvec on the tensor cores, for several activation rows
// (speculative verification: one token plus drafts, M up to 16).
//
// The per-pair fp16 FMA of the matvec kernel in gemv.cu costs one instruction
// per activation row, so its time grows with M. Here the decoded weights feed
// mma.sync.m16n8k16 (fp16 operands, fp32 accumulation) as the A operand
// straight from registers, with the activations as B (n = activation row, one
// or two n8 tiles): the decode costs the same as for one row and the
// contraction over M runs on the tensor pipe.
//
// Work split. Tiles are 16 rows (one row group of the packed record layout),
// numbered across the tasks of a batch; each CTA takes a contiguous range of
// about equal bytes. Within a CTA all 16 consumer warps work on every step
// (1024 columns) of a tile: warp w takes 64 columns (half of block w/2), so
// each warp issues 4 MMAs per step and n-tile, and the CTA never waits on a
// ragged split of steps between warps. Partial sums of the 16 warps meet in
// shared memory (fp32 atomics); the last warp to add writes y.
//
// Streaming. A producer warp copies each step of a tile into a ring slot:
// one 1D bulk copy per row (16 per slot) into rows padded to 272 B (ternary)
// or 544 B (INT4), so that the 8 rows one load instruction touches fall on
// distinct shared-memory banks. Full barriers complete on the copies' byte
// count, empty barriers on one arrival per consumer warp. All waits are
// bounded and record QMV_ERR_TIMEOUT in the device error word.
//
// MMA operand mapping. Lane (g, t) = (lane / 4, lane % 4) holds A rows g and
// g + 8 and B column n = g. Any bijection between the MMA's k index and the
// columns works as long as A and B agree; here lane t's A entries of the four
// k-slices of a warp's 64 columns are the 16 columns 16t..16t+15 (pair i =
// columns 2i, 2i+1 of that run): k-slice j takes pair 2j at k = 2t, 2t+1 and
// pair 2j+1 at k = 2t+8, 2t+9. These 16 columns are one ternary code word (or
// two INT4 words) of a row, decoded with the fixed shifts of gemv_core.cuh, and
// the lane's B registers are the activation pairs of the same columns, i.e.
// 32 contiguous bytes of staged x.
//
// Block scales. Each k-slice lies inside one 128-column block, so the warp's
// four MMAs accumulate one block-half; the fp32 result is scaled by the
// block's fp16 scale of row g / g + 8 and added to the running sum. Ternary
// codes decode to v = 1 + q/2 (see gemv.cu); the accumulator starts at
// -sum(x) of the block-half, leaving (1/2) sum q x, and the factor 2 is applied
// when y is written. INT4 decodes to q exactly.
//
// Activations are staged per chunk of K as fp16, scaled per row by a power of
// two (largest magnitude in [2^9, 2^10) for ternary, [2^8, 2^9) for INT4), in
// 16-byte units whose index is XORed with (row & 7) so that the 32 lanes of a
// load hit all banks.
#include <algorithm>

#include "gemv_core.cuh"

namespace qmv {
namespace {

using namespace core;

constexpr int kMmaWarps = 16;                        // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;    // + one producer warp
constexpr int kTileRows = 16;

template <int FMT>
struct MmaGeo {
  static constexpr int WPB = Fmt<FMT>::WPB;
  static constexpr int BLOCK_BYTES = WPB * 4;
  static constexpr int ROW_STEP = kBlocksPerStep * BLOCK_BYTES;       // 256 / 512
  static constexpr int PITCH = ROW_STEP + (FMT == QMV_TERNARY2 ? 16 : 32);  // row pitch in the ring
  static constexpr int SLOT = kTileRows * PITCH;
  static constexpr int RING = FMT == QMV_TERNARY2 ? 8 : 5;            // slots
  static constexpr int NBUF = RING + 2;                               // reduction buffers
};

__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(kMmaWarps * 32) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ int find_task_mma(const GemvBatch& b, int tile) {
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Walks a CTA's (tile, chunk, step) sequence in the order both the producer and
// the consumers use: per task segment of the tile range, chunk by chunk, every
// tile of the segment, every step of the chunk.
struct Walk {
  int tile, seg_begin, seg_end, ti, kc0, s, N, K, nb, nsteps;
  __device__ bool start(const GemvBatch& b, int tile_begin, int tile_end, int KC) {
    tile = seg_begin = tile_begin;
    if (tile >= tile_end) return false;
    begin_segment(b, tile_end, KC);
    return true;
  }
  __device__ void begin_segment(const GemvBatch& b, int tile_end, int KC) {
    ti = find_task_mma(b, seg_begin);
    N = b.t[ti].N;
    K = b.t[ti].K;
    seg_end = min(tile_end, b.t[ti].tile0 + (N + kTileRows - 1) / kTileRows);
    tile = seg_begin;
    kc0 = 0;
    s = 0;
    nb = min(KC, K) / 128;
    nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;
  }
  // advance one step; returns false at the end of the CTA's range
  __device__ bool next(const GemvBatch& b, int tile_end, int KC) {
    if (++s < nsteps) return true;
    s = 0;
    if (++tile < seg_end) return true;
    tile = seg_begin;
    kc0 += KC;
    if (kc0 < K) {
      nb = min(KC, K - kc0) / 128;
      nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;
      return true;
    }
    seg_begin = seg_end;
    if (seg_begin >= tile_end) return false;
    begin_segment(b, tile_end, KC);
    return true;
  }
};

// Stage columns [kc0, kc0 + kcn) of the M activation rows (MT >= M slots; the
// rest zero) and, for ternary, -sum(x) of every 64-column half-block.
template <int FMT, int MT>
__device__ void stage_mma(const uint16_t* __restrict__ x, int ldx, int kc0, int kcn, int M, int KCU, uint4* xs,
                          float* xneg, float (*s_red)[MT], float* s_xinv) {
  using F = Fmt<FMT>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int NT = kMmaWarps * 32;
  const int nu = kcn / 8;  // 16-byte units per row
  bar_consumers();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float mx = 0.f;
    if (m < M)
      for (int u = tid; u < nu; u += NT) {
        const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)m * ldx + kc0 + u * 8);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t w = word_of(raw, e);
          mx = fmaxf(mx, fmaxf(fabsf(bf16_to_f32(w & 0xFFFFu)), fabsf(bf16_to_f32(w >> 16))));
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp][m] = mx;
  }
  bar_consumers();
  __shared__ float s_xscale[MT];
  if (tid < MT) {
    float mx = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) mx = fmaxf(mx, s_red[w][tid]);
    int e = 0;
    if (mx > 0.f && mx <= 3.4e38f) {
      int ex;
      frexpf(mx, &ex);
      e = max(-120, min(120, F::XLOG2 - (ex - 1)));
    }
    s_xscale[tid] = exp2i(e);
    s_xinv[tid] = exp2i(-e);
  }
  bar_consumers();
  for (int q = tid; q < MT * nu; q += NT) {
    const int m = q / nu, u = q - m * nu;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (m < M) {
      const float sc = s_xscale[m];
      const uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)m * ldx + kc0 + u * 8);
      uint32_t hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = word_of(raw, e);
        hv[e] = h2u(__floats2half2_rn(bf16_to_f32(w & 0xFFFFu) * sc, bf16_to_f32(w >> 16) * sc));
      }
      out = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
    xs[(size_t)m * KCU + (u ^ (m & 7))] = out;
  }
  if constexpr (FMT == QMV_TERNARY2) {
    bar_consumers();
    const int nh = kcn / 64;
    for (int q = tid; q < nh * MT; q += NT) {
      const int hb = q / MT, m = q - hb * MT;
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 v = xs[(size_t)m * KCU + ((hb * 8 + u) ^ (m & 7))];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(as_h2(word_of(v, e)));
          sum += f.x + f.y;
        }
      }
      xneg[q] = -sum;
    }
  }
  bar_consumers();
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const __grid_constant__ GemvBatch b, int M) {
  using F = Fmt<FMT>;
  using G = MmaGeo<FMT>;
  constexpr int MT = 8 * NT;
  constexpr bool TERN = FMT == QMV_TERNARY2;
  constexpr int R = G::RING;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;                                              // [R][16][PITCH]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + R * G::SLOT);       // [R]
  uint64_t* empty = full + R;                                                  // [R]
  float* red = reinterpret_cast<float*>(empty + R);                            // [NBUF][16][MT]
  int* cnt = reinterpret_cast<int*>(red + G::NBUF * kTileRows * MT);           // [NBUF] (+pad)
  const int KC = b.kc;
  const int KCU = KC / 8;
  uint4* xs = reinterpret_cast<uint4*>(cnt + 32);                              // [MT][KCU]
  float* xneg = reinterpret_cast<float*>(xs + (size_t)MT * KCU);               // [KC/64][MT]
  __shared__ float s_red[kMmaWarps][MT];
  __shared__ float s_xinv[MT];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile_begin = b.cta_tile[blockIdx.x];
  const int tile_end = b.cta_tile[blockIdx.x + 1];

  if (tid == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMmaWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < G::NBUF * kTileRows * MT; i += kMmaThreads) red[i] = 0.f;
  if (tid < G::NBUF) cnt[tid] = 0;
  __syncthreads();

  if (warp == kMmaWarps) {
    // ===================== producer warp: one bulk copy per row of each step
    Walk wk;
    if (!wk.start(b, tile_begin, tile_end, KC)) return;
    uint32_t it = 0;
    do {
      const int slot = it % R;
      if (it >= (uint32_t)R) mbar_wait(&empty[slot], ((it / R) - 1) & 1u, b.err);
      const GemvTask& T = b.t[wk.ti];
      const int nbk = min(kBlocksPerStep, wk.nb - wk.s * kBlocksPerStep);
      const uint32_t row_bytes = (uint32_t)nbk * G::BLOCK_BYTES;
      const int group = wk.tile - T.tile0;  // 16-row group within the matrix
      const unsigned char* src = reinterpret_cast<const unsigned char*>(T.codes) +
                                 (size_t)group * kTileRows * (T.K / F::CPW) * 4 +
                                 (size_t)(wk.kc0 / kStep + wk.s) * kTileRows * G::ROW_STEP;
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&full[slot], kTileRows * row_bytes);
      }
      __syncwarp();
      if (lane < kTileRows)
        bulk_g2s(ring + (size_t)slot * G::SLOT + lane * G::PITCH, src + (size_t)lane * row_bytes, row_bytes,
                 &full[slot]);
      __syncwarp();
      ++it;
    } while (wk.next(b, tile_end, KC));
    return;
  }

  // ===================== consumer warps
  const int g = lane >> 2, t = lane & 3;
  const int bw = warp >> 1, hw = warp & 1;  // block of the step, half of the block
  const DecodeK dk = load_decode_k(b.magic);
  Walk wk;
  if (!wk.start(b, tile_begin, tile_end, KC)) return;
  uint32_t it = 0, unit = 0;
  const uint16_t* staged_x = nullptr;
  int staged_kc0 = -1, staged_K = -1;
  float tot[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) tot[n][e] = 0.f;

  do {
    const GemvTask& T = b.t[wk.ti];
    if (wk.tile == wk.seg_begin && wk.s == 0) {
      // first step of a chunk for this segment: stage its activations
      if (T.x != staged_x || wk.kc0 != staged_kc0 || wk.K != staged_K) {
        stage_mma<FMT, MT>(T.x, T.ldx, wk.kc0, min(KC, wk.K - wk.kc0), M, KCU, xs, xneg, s_red, s_xinv);
        staged_x = T.x;
        staged_kc0 = wk.kc0;
        staged_K = wk.K;
      }
    }
    const int nbk = min(kBlocksPerStep, wk.nb - wk.s * kBlocksPerStep);
    const int row0 = (wk.tile - T.tile0) * kTileRows;
    const int slot = it % R;
    // scales of rows g, g+8 for this warp's block (rows past N read the last row; never stored)
    unsigned short sg = 0, sg8 = 0;
    const bool active = bw < nbk;
    const int blk = wk.kc0 / 128 + wk.s * kBlocksPerStep + bw;
    if (active) {
      const int KB = wk.K / 128;
      sg = __ldg(reinterpret_cast<const unsigned short*>(T.scales) + (size_t)min(row0 + g, wk.N - 1) * KB + blk);
      sg8 = __ldg(reinterpret_cast<const unsigned short*>(T.scales) + (size_t)min(row0 + g + 8, wk.N - 1) * KB + blk);
    }
    mbar_wait(&full[slot], (it / R) & 1u, b.err);
    if (active) {
      const unsigned char* rows = ring + (size_t)slot * G::SLOT;
      // this lane's 16 columns of rows g and g+8
      uint32_t wg[TERN ? 1 : 2], wg8[TERN ? 1 : 2];
      if constexpr (TERN) {
        const int wo = (bw * 8 + hw * 4 + t) * 4;
        wg[0] = *reinterpret_cast<const uint32_t*>(rows + g * G::PITCH + wo);
        wg8[0] = *reinterpret_cast<const uint32_t*>(rows + (g + 8) * G::PITCH + wo);
      } else {
        const int wo = (bw * 16 + hw * 8 + 2 * t) * 4;
        const uint2 a = *reinterpret_cast<const uint2*>(rows + g * G::PITCH + wo);
        const uint2 c = *reinterpret_cast<const uint2*>(rows + (g + 8) * G::PITCH + wo);
        wg[0] = a.x; wg[1] = a.y;
        wg8[0] = c.x; wg8[1] = c.y;
      }
      // decode: pair p (columns 2p, 2p+1 of the lane's 16) of rows g / g+8
      uint32_t ag[8], ag8[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if constexpr (TERN) {
          ag[p] = h2u(decode_pair<FMT>(wg[0], p, dk));
          ag8[p] = h2u(decode_pair<FMT>(wg8[0], p, dk));
        } else {
          ag[p] = h2u(decode_pair<FMT>(wg[p >> 2], p & 3, dk));
          ag8[p] = h2u(decode_pair<FMT>(wg8[p >> 2], p & 3, dk));
        }
      }
      const float fg = __half2float(__ushort_as_half(sg));
      const float fg8 = __half2float(__ushort_as_half(sg8));
      const int u0 = wk.s * 128 + bw * 16 + hw * 8 + 2 * t;  // staged 16-byte unit of the lane's first 8 columns
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int m = n * 8 + g;
        const uint4 x0 = xs[(size_t)m * KCU + (u0 ^ g)];
        const uint4 x1 = xs[(size_t)m * KCU + ((u0 + 1) ^ g)];
        const uint32_t xp[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float d[4];
        if constexpr (TERN) {
          const float2 xn = *reinterpret_cast<const float2*>(xneg + (size_t)(wk.s * 16 + bw * 2 + hw) * MT + n * 8 + 2 * t);
          d[0] = xn.x; d[1] = xn.y; d[2] = xn.x; d[3] = xn.y;
        } else {
          d[0] = d[1] = d[2] = d[3] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a[4] = {ag[2 * j], ag8[2 * j], ag[2 * j + 1], ag8[2 * j + 1]};
          mma16816(d, a, xp[2 * j], xp[2 * j + 1]);
        }
        tot[n][0] = fmaf(d[0], fg, tot[n][0]);
        tot[n][1] = fmaf(d[1], fg, tot[n][1]);
        tot[n][2] = fmaf(d[2], fg8, tot[n][2]);
        tot[n][3] = fmaf(d[3], fg8, tot[n][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    ++it;

    if (wk.s == wk.nsteps - 1) {
      // ---- end of this tile's chunk: combine the 16 warps' partial sums
      float* buf = red + (size_t)(unit % G::NBUF) * kTileRows * MT;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int c0 = n * 8 + 2 * t;
        atomicAdd(&buf[g * MT + c0], tot[n][0]);
        atomicAdd(&buf[g * MT + c0 + 1], tot[n][1]);
        atomicAdd(&buf[(g + 8) * MT + c0], tot[n][2]);
        atomicAdd(&buf[(g + 8) * MT + c0 + 1], tot[n][3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) tot[n][e] = 0.f;
      }
      __syncwarp();
      int old = 0;
      if (lane == 0) {
        __threadfence_block();
        old = atomicAdd(&cnt[unit % G::NBUF], 1);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == kMmaWarps - 1) {
        __threadfence_block();
        constexpr float kFactor = TERN ? 2.f : 1.f;
        const bool first = wk.kc0 == 0;
        for (int e = lane; e < kTileRows * MT; e += 32) {
          const int r = e / MT, m = e - r * MT;
          const float v = buf[e];
          buf[e] = 0.f;
          const int row = row0 + r;
          if (row < wk.N && m < M) {
            float* yp = T.y + (size_t)m * T.ldy + row;
            const float val = kFactor * v * s_xinv[m];
            *yp = first ? val : *yp + val;
          }
        }
        __syncwarp();
        if (lane == 0) cnt[unit % G::NBUF] = 0;
        __syncwarp();
      }
      ++unit;
    }
  } while (wk.next(b, tile_end, KC));
}

template <int FMT, int NT>
int launch_mma_t(GemvBatch& b, int M, cudaStream_t s) {
  using G = MmaGeo<FMT>;
  constexpr int MT = 8 * NT;
  constexpr size_t kSmemMax = 227 * 1024;
  int tiles = 0, max_K = 0;
  for (int i = 0; i < b.n_tasks; ++i) {
    b.t[i].tile0 = tiles;
    tiles += (b.t[i].N + kTileRows - 1) / kTileRows;
    max_K = std::max(max_K, (int)b.t[i].K);
  }
  b.n_tiles = tiles;
  b.rows_per_tile = kTileRows;
  const size_t ring = (size_t)G::RING * G::SLOT + 2 * G::RING * 8 + (size_t)G::NBUF * kTileRows * MT * 4 + 32 * 4;
  const size_t budget = kSmemMax - ring - 2048;  // static shared memory (s_red, s_xinv, s_xscale) < 2 KB
  // per staged column: MT fp16 values, and for ternary MT floats per 64 columns
  const size_t per_col = (size_t)MT * 2 + (FMT == QMV_TERNARY2 ? ((size_t)MT * 4 + 63) / 64 : 0);
  int kc = (int)(budget / per_col) / kStep * kStep;
  const int need = (max_K + kStep - 1) / kStep * kStep;
  if (kc > need) kc = need;
  if (kc < kStep) return fail(QMV_ERR_UNSUPPORTED, "activation chunk does not fit shared memory for M=%d", M);
  b.kc = kc;
  const size_t smem = ring + (size_t)MT * kc * 2 + (FMT == QMV_TERNARY2 ? (size_t)(kc / 64) * MT * 4 : 0);
  fill_magic<FMT>(b.magic);
  b.err = device_error_word();
  if (!b.err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  auto kern = gemv_mma_kernel<FMT, NT>;
  int per_sm = 0;
  int rc = kernel_fit((const void*)kern, kMmaThreads, smem, &per_sm);
  if (rc != QMV_OK) return rc;
  const int grid = std::min(std::min(sm_count(), kMaxCtas), tiles);
  double total = 0;
  for (int i = 0; i < b.n_tasks; ++i) total += (double)((b.t[i].N + 15) / 16 * 16) * b.t[i].K;
  b.n_ctas = grid;
  b.cta_tile[0] = 0;
  int c = 1;
  double done = 0;
  for (int i = 0; i < b.n_tasks && c < grid; ++i) {
    const int nt = (b.t[i].N + kTileRows - 1) / kTileRows;
    for (int j = 0; j < nt && c < grid; ++j) {
      done += (double)kTileRows * b.t[i].K;
      while (c < grid && done >= total * c / grid) b.cta_tile[c++] = b.t[i].tile0 + j + 1;
    }
  }
  for (; c <= grid; ++c) b.cta_tile[c] = tiles;
  kern<<<grid, kMmaThreads, smem, s>>>(b, M);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(QMV_ERR_CUDA, "gemv (tensor-core) launch of %d CTAs x %d threads, %zu B shared memory, %d tiles, chunk %d: %s",
                grid, kMmaThreads, smem, tiles, kc, cudaGetErrorString(e));
  return QMV_OK;
}

}  // namespace

int launch_gemv_mma(int format, GemvBatch& b, int M, cudaStream_t s) {
  if (M < 1 || M > 16) return fail(QMV_ERR_ARG, "M=%d outside 1..16 for one launch", M);
  if (format == QMV_TERNARY2) return M <= 8 ? launch_mma_t<QMV_TERNARY2, 1>(b, M, s) : launch_mma_t<QMV_TERNARY2, 2>(b, M, s);
  if (format == QMV_INT4) return M <= 8 ? launch_mma_t<QMV_INT4, 1>(b, M, s) : launch_mma_t<QMV_INT4, 2>(b, M, s);
  return fail(QMV_ERR_UNSUPPORTED, "format %d has no tensor-core matvec kernel", format);
}

}  // namespace qmv
