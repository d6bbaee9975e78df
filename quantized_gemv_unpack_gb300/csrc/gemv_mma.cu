// Fused dequantize-and-matvec on the tensor cores, for several activation rows
// (speculative verification: one token plus drafts, M up to 16).
//
// The per-pair fp16 FMA of the matvec kernel in gemv.cu costs one instruction
// per activation row, so its time grows with M. Here the decoded weights feed
// mma.sync.m16n8k16 (bf16 operands, fp32 accumulation) as the A operand
// straight from registers, with the activations as B (n = activation row, one
// or two n8 tiles): the decode costs the same as for one row and the
// contraction over M runs on the tensor pipe.
//
// Work split. Tiles are 16 rows (one row group of the packed record layout),
// numbered across the tasks of a batch; each CTA takes a contiguous range of
// about equal bytes. A CTA runs four independent pipelines ("quads" of 4
// warps, one warp per SM sub-partition): per task segment and activation chunk,
// quad q takes every 4th tile from the q-th, and its warp w takes blocks 2w and
// 2w + 1 of every 1024-column step of those tiles (16 MMAs per step and n-tile).
// At the end of a tile's chunk the quad's four partial sums meet in shared
// memory behind a 128-thread barrier and are added in a fixed order, so results
// are reproducible bit for bit. The whole CTA synchronises only to restage
// activations.
//
// Streaming. Each step of a tile is one contiguous code record of the packed
// layout (16 rows x 1024 columns, 4 KB ternary / 8 KB INT4) plus its 256-byte
// scale record; both land in a slot of the quad's ring (4 slots ternary, 3
// INT4) with one 1D bulk copy each. The copy duty rotates over the quad's warps:
// after step i, warp i % 4 refills the slot of step i - 1 with step i + RING - 1
// once the quad is done with step i - 1. Full barriers complete on the copies'
// byte count, empty barriers on one arrival per warp of the quad. All waits are
// bounded and record QMV_ERR_TIMEOUT in the device error word.
//
// MMA operand mapping. Lane (g, t) = (lane / 4, lane % 4) holds A rows g and
// g + 8 and B column n = g. Any bijection between the MMA's k index and the
// columns works as long as A and B agree; here lane t's A entries of the eight
// k-slices of a 128-column block are the 32 columns 32t..32t+31 (pair p =
// columns 32t + 2p, +1): k-slice j takes pair 2j at k = 2t, 2t+1 and pair
// 2j+1 at k = 2t+8, 2t+9. These 32 columns are two ternary code words (or four
// INT4 words) of a row, and the lane's B registers are the activation pairs of
// the same columns, i.e. 64 contiguous bytes of staged x. The 8 rows one code load touches share banks
// (rows are 256 or 512 B apart in a slot); those loads stay well below the
// shared-memory bandwidth.
//
// Operands are bf16 (mma.sync m16n8k16, bf16 x bf16 -> fp32). The activations
// are the caller's bf16 values, copied unchanged into shared memory, so there is
// no range limit and no rounding before the products. The weights decode to
// bf16 exactly: ternary codes, shifted to bits 6-7 / 22-23, give
// (t & 0x00C000C0) ^ 0x3F803F80 = 1 + q/2 (bit 6 is the mantissa MSB, bit 7 the
// exponent LSB of bf16 1.0), and subtracting 1.0 leaves q/2 (a zero code is an
// exact 0); INT4 nibbles give (t & 0x000F000F) ^ 0x43084308 = 136 + q (128 plus
// the offset-binary nibble), and subtracting 136 leaves q. Every product is
// exact in fp32 and only the fp32 accumulation rounds.
//
// Block scales. Each k-slice lies inside one 128-column block, so a warp's
// eight MMAs of a block accumulate that block; the fp32 result is scaled by
// the block's fp16 scale of row g / g + 8 (from the scale record in the slot)
// and added to the running sum. Ternary sums carry q/2, so the factor 2 is
// applied when y is written.
//
// Activations are staged per chunk of K in 16-byte units whose index is XORed
// with (row & 7) so that the 32 lanes of a load hit all banks.
#include <algorithm>

#include "gemv_core.cuh"

namespace qmv {
namespace {

using namespace core;

constexpr int kMmaWarps = 16;                        // warps per CTA
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kQuads = 4;                            // independent 4-warp pipelines per CTA
constexpr int kTileRows = 16;

template <int FMT>
struct MmaGeo {
  static constexpr int WPB = Fmt<FMT>::WPB;
  static constexpr int BLOCK_BYTES = WPB * 4;
  static constexpr int ROW_STEP = kBlocksPerStep * BLOCK_BYTES;       // 256 / 512
  static constexpr int SLOT = kTileRows * ROW_STEP;                   // one record: 4 / 8 KB
  static constexpr int RING = FMT == QMV_TERNARY2 ? 4 : 3;            // slots per quad (64 / 96 KB per CTA)
};

__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(kMmaWarps * 32) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16 decode constants (kernel parameters, so they live in registers and the
// shifts keep their unit): mask, base (also the value subtracted), the left
// shift multipliers 2^6, 2^4, 2^2 and the right shift amounts 2, 4, 6, 8
// (ternary) or, for INT4, right shifts 4, 8, 12 in r2, r4, r6.
struct DecodeB {
  uint32_t mask, base, m6, m4, m2, r2, r4, r6, r8;
};
template <int FMT>
inline void fill_magic_bf16(uint32_t* magic) {
  const bool tern = FMT == QMV_TERNARY2;
  magic[0] = tern ? 0x00C000C0u : 0x000F000Fu;
  magic[1] = tern ? 0x3F803F80u : 0x43084308u;
  magic[2] = 1u << 6;
  magic[3] = 1u << 4;
  magic[4] = 1u << 2;
  magic[5] = tern ? 2 : 4;
  magic[6] = tern ? 4 : 8;
  magic[7] = tern ? 6 : 12;
  magic[8] = 8;
  magic[9] = 0;
}
__device__ __forceinline__ DecodeB load_decode_b(const uint32_t* m) {
  return DecodeB{m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], m[8]};
}
// Column pair i of code word w as two exact bf16 weights: ternary q/2, INT4 q.
template <int FMT>
__device__ __forceinline__ uint32_t decode_pair_bf16(uint32_t w, int i, const DecodeB& k) {
  uint32_t t;
  if constexpr (FMT == QMV_TERNARY2) {
    // pair i's codes at bits 2i..2i+1 and 16+2i..17+2i, moved to bits 6-7 / 22-23
    switch (i) {
      case 0: t = mul_lo(w, k.m6); break;
      case 1: t = mul_lo(w, k.m4); break;
      case 2: t = mul_lo(w, k.m2); break;
      case 3: t = w; break;
      case 4: t = shr_r(w, k.r2); break;
      case 5: t = shr_r(w, k.r4); break;
      case 6: t = shr_r(w, k.r6); break;
      default: t = shr_r(w, k.r8); break;
    }
  } else {
    t = i == 0 ? w : shr_r(w, i == 1 ? k.r2 : (i == 2 ? k.r4 : k.r6));
  }
  return sub_bf16x2(and_xor(t, k.mask, k.base), k.base);
}

__device__ __forceinline__ int find_task_mma(const GemvBatch& b, int tile) {
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Walks one quad's (tile, chunk, step) sequence: per task segment of the CTA's
// tile range, chunk by chunk, the quad's tiles of the segment (every 4th, from
// the quad's index), every step of the chunk.
struct QuadWalk {
  int seg_begin, seg_end, ti, K, kc0, nb, nsteps, tile, s, q;
  __device__ bool start(const GemvBatch& b, int tile_begin, int tile_end, int KC, int quad) {
    q = quad;
    seg_begin = tile_begin;
    if (seg_begin >= tile_end) return false;
    begin_segment(b, tile_end, KC);
    return settle(b, tile_end, KC);
  }
  __device__ void begin_segment(const GemvBatch& b, int tile_end, int KC) {
    ti = find_task_mma(b, seg_begin);
    K = b.t[ti].K;
    seg_end = min(tile_end, b.t[ti].tile0 + (b.t[ti].N + kTileRows - 1) / kTileRows);
    kc0 = 0;
    begin_chunk(KC);
  }
  __device__ void begin_chunk(int KC) {
    nb = min(KC, K - kc0) / 128;
    nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;
    tile = seg_begin + q;
    s = 0;
  }
  // move past segment-chunks in which this quad has no tile; false at the end
  __device__ bool settle(const GemvBatch& b, int tile_end, int KC) {
    while (tile >= seg_end) {
      kc0 += KC;
      if (kc0 < K) {
        begin_chunk(KC);
        continue;
      }
      seg_begin = seg_end;
      if (seg_begin >= tile_end) return false;
      begin_segment(b, tile_end, KC);
    }
    return true;
  }
  __device__ bool next(const GemvBatch& b, int tile_end, int KC) {
    if (++s < nsteps) return true;
    s = 0;
    tile += kQuads;
    return settle(b, tile_end, KC);
  }
};

// Stage columns [kc0, kc0 + kcn) of the M activation rows: the bf16 values
// unchanged, 16-byte unit u of row m at m * KCU + (u ^ (m & 7)).
__device__ void stage_mma(const uint16_t* __restrict__ x, int ldx, int kc0, int kcn, int M, int KCU, uint4* xs) {
  const int tid = threadIdx.x;
  constexpr int NT = kMmaWarps * 32;
  const int nu = kcn / 8;  // 16-byte units per row
  bar_consumers();
  for (int q = tid; q < M * nu; q += NT) {
    const int m = q / nu, u = q - m * nu;
    xs[(size_t)m * KCU + (u ^ (m & 7))] = *reinterpret_cast<const uint4*>(x + (size_t)m * ldx + kc0 + u * 8);
  }
  bar_consumers();
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const __grid_constant__ GemvBatch b, int M) {
  using F = Fmt<FMT>;
  using G = MmaGeo<FMT>;
  constexpr int MT = 8 * NT;
  constexpr bool TERN = FMT == QMV_TERNARY2;
  constexpr int R = G::RING;  // slots per quad

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;                                                          // [4][R][SLOT]
  unsigned short* sring = reinterpret_cast<unsigned short*>(smem_raw + kQuads * R * G::SLOT);  // [4][R][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(sring + kQuads * R * 128);                  // [4][R]
  uint64_t* empty = full + kQuads * R;                                                     // [4][R]
  float* red = reinterpret_cast<float*>(empty + kQuads * R);                               // [4][2][4][16][MT]
  const int KC = b.kc;
  const int KCU = KC / 8;
  uint4* xs = reinterpret_cast<uint4*>(red + kQuads * 2 * 4 * kTileRows * MT);             // [M][KCU]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp >> 2, wq = warp & 3;  // quad, and position in it
  const int tile_begin = b.cta_tile[blockIdx.x];
  const int tile_end = b.cta_tile[blockIdx.x + 1];
  unsigned char* qring = ring + (size_t)quad * R * G::SLOT;
  unsigned short* qsring = sring + (size_t)quad * R * 128;
  uint64_t* qfull = full + quad * R;
  uint64_t* qempty = empty + quad * R;
  float* qred = red + (size_t)quad * 2 * 4 * kTileRows * MT;

  if (b.test_wait_us && test_wait_times_out(b.err, b.test_wait_us)) return;
  if (tid < kQuads * R) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 4);
  }
  if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  if (tile_begin >= tile_end) return;

  // ---- streaming: step i of this quad's sequence lands in slot i % R of the
  // quad's ring as two bulk copies, its code record and its scale record. The
  // copies of step i + R - 1 are issued by warp i % 4 of the quad right after it
  // finished step i, once the quad is done with step i - 1 (whose slot they
  // reuse); steps 0 .. R-2 are issued up front.
  auto issue_step = [&](const QuadWalk& w, uint32_t step) {
    const GemvTask& T = b.t[w.ti];
    const int nbk = min(kBlocksPerStep, w.nb - w.s * kBlocksPerStep);
    const uint32_t bytes = (uint32_t)(kTileRows * nbk * G::BLOCK_BYTES);
    const size_t grp = (size_t)(w.tile - T.tile0);
    const size_t st = (size_t)(w.kc0 / kStep + w.s);
    const unsigned char* src = reinterpret_cast<const unsigned char*>(T.codes) + grp * kTileRows * (T.K / F::CPW) * 4 +
                               st * kTileRows * G::ROW_STEP;
    const int slot = step % R;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of the slot precede the copy
    mbar_arrive_expect_tx(&qfull[slot], bytes + 256u);
    bulk_g2s(qring + (size_t)slot * G::SLOT, src, bytes, &qfull[slot]);
    bulk_g2s(qsring + (size_t)slot * 128, T.scales + (grp * scale_steps(T.K) + st) * 128, 256u, &qfull[slot]);
  };
  QuadWalk pw;  // position of step it + R - 1 of this quad
  bool pw_live = pw.start(b, tile_begin, tile_end, KC, quad);
  for (int i = 0; i < R - 1 && pw_live; ++i) {
    if (wq == 0 && lane == 0) issue_step(pw, i);
    pw_live = pw.next(b, tile_end, KC);
  }

  const int g = lane >> 2, t = lane & 3;
  const DecodeB dk = load_decode_b(b.magic);
  const uint16_t* staged_x = nullptr;
  int staged_kc0 = -1, staged_K = -1;
  uint32_t it = 0, tile_no = 0;

  // segment-chunks in CTA order: every warp stages each one (the barrier inside
  // needs all 16), then the quad works through its tiles of it
  int seg_begin = tile_begin;
  while (seg_begin < tile_end) {
    const int ti = find_task_mma(b, seg_begin);
    const GemvTask& T = b.t[ti];
    const int N = T.N, K = T.K;
    const int seg_end = min(tile_end, T.tile0 + (N + kTileRows - 1) / kTileRows);
    for (int kc0 = 0; kc0 < K; kc0 += KC) {
      const int kcn = min(KC, K - kc0);
      if (T.x != staged_x || kc0 != staged_kc0 || K != staged_K) {
        stage_mma(T.x, T.ldx, kc0, kcn, M, KCU, xs);
        staged_x = T.x;
        staged_kc0 = kc0;
        staged_K = K;
      }
      const int nb = kcn / 128;
      const int nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;
      for (int tile = seg_begin + quad; tile < seg_end; tile += kQuads, ++tile_no) {
        float tot[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) tot[n][e] = 0.f;
        for (int s = 0; s < nsteps; ++s, ++it) {
          const int nbk = min(kBlocksPerStep, nb - s * kBlocksPerStep);
          const int slot = it % R;
          mbar_wait(&qfull[slot], (it / R) & 1u, b.err);
          const unsigned char* rows = qring + (size_t)slot * G::SLOT;
          const int row_bytes = nbk * G::BLOCK_BYTES;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int bk = wq * 2 + j;  // block of the step
            if (bk >= nbk) break;
            // this lane's 32 columns (32t .. 32t+31 of the block) of rows g and g+8
            uint32_t wg[TERN ? 2 : 4], wg8[TERN ? 2 : 4];
            if constexpr (TERN) {
              const int wo = bk * G::BLOCK_BYTES + t * 8;
              const uint2 a = *reinterpret_cast<const uint2*>(rows + g * row_bytes + wo);
              const uint2 c = *reinterpret_cast<const uint2*>(rows + (g + 8) * row_bytes + wo);
              wg[0] = a.x; wg[1] = a.y;
              wg8[0] = c.x; wg8[1] = c.y;
            } else {
              const int wo = bk * G::BLOCK_BYTES + t * 16;
              const uint4 a = *reinterpret_cast<const uint4*>(rows + g * row_bytes + wo);
              const uint4 c = *reinterpret_cast<const uint4*>(rows + (g + 8) * row_bytes + wo);
              wg[0] = a.x; wg[1] = a.y; wg[2] = a.z; wg[3] = a.w;
              wg8[0] = c.x; wg8[1] = c.y; wg8[2] = c.z; wg8[3] = c.w;
            }
            const float fg = __half2float(__ushort_as_half(qsring[(size_t)slot * 128 + g * 8 + bk]));
            const float fg8 = __half2float(__ushort_as_half(qsring[(size_t)slot * 128 + (g + 8) * 8 + bk]));
            const int u0 = s * 128 + bk * 16 + 4 * t;  // staged 16-byte unit of the lane's first 8 columns
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              // lanes of activation rows past M load row n*8 instead (the same address as
              // a live lane, so no extra shared-memory traffic); their output columns are
              // never stored
              const int m = n * 8 + g < M ? n * 8 + g : n * 8;
              uint32_t xp[16];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint4 xv = xs[(size_t)m * KCU + ((u0 + v) ^ (m & 7))];
                xp[4 * v] = xv.x; xp[4 * v + 1] = xv.y; xp[4 * v + 2] = xv.z; xp[4 * v + 3] = xv.w;
              }
              float d[4] = {0.f, 0.f, 0.f, 0.f};
              // odd k-slices accumulate apart (two independent MMA chains per block)
              float d2[4] = {0.f, 0.f, 0.f, 0.f};
              // k-slice kk: pairs 2kk and 2kk+1 (columns 32t + 4kk .. +3) of rows g and g+8
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                constexpr int PPW = F::PPW;
                const int p0 = 2 * kk, p1 = 2 * kk + 1;
                const uint32_t a[4] = {decode_pair_bf16<FMT>(wg[p0 / PPW], p0 % PPW, dk),
                                       decode_pair_bf16<FMT>(wg8[p0 / PPW], p0 % PPW, dk),
                                       decode_pair_bf16<FMT>(wg[p1 / PPW], p1 % PPW, dk),
                                       decode_pair_bf16<FMT>(wg8[p1 / PPW], p1 % PPW, dk)};
                if (kk & 1) mma16816(d2, a, xp[2 * kk], xp[2 * kk + 1]);
                else mma16816(d, a, xp[2 * kk], xp[2 * kk + 1]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) d[e] += d2[e];
              tot[n][0] = fmaf(d[0], fg, tot[n][0]);
              tot[n][1] = fmaf(d[1], fg, tot[n][1]);
              tot[n][2] = fmaf(d[2], fg8, tot[n][2]);
              tot[n][3] = fmaf(d[3], fg8, tot[n][3]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[slot]);
          // refill: step it + R - 1 of the quad goes to the slot of step it - 1, issued by warp it % 4
          if (pw_live) {
            if (wq == (int)(it % 4)) {
              if (it >= 1) mbar_wait(&qempty[(it - 1) % R], ((it - 1) / R) & 1u, b.err);
              if (lane == 0) issue_step(pw, it + R - 1);
            }
            pw_live = pw.next(b, tile_end, KC);
          }
        }
        // ---- end of this tile's chunk: the quad's 4 partial sums, added in a fixed order
        float* buf = qred + (size_t)(tile_no & 1) * 4 * kTileRows * MT;
        float* mine = buf + (size_t)wq * kTileRows * MT;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int c0 = n * 8 + 2 * t;
          *reinterpret_cast<float2*>(&mine[g * MT + c0]) = make_float2(tot[n][0], tot[n][1]);
          *reinterpret_cast<float2*>(&mine[(g + 8) * MT + c0]) = make_float2(tot[n][2], tot[n][3]);
        }
        asm volatile("bar.sync %0, 128;" ::"r"(2 + quad) : "memory");
        if (wq == (int)(tile_no & 3)) {  // the writing warp rotates
          constexpr float kFactor = TERN ? 2.f : 1.f;
          const int row0 = (tile - T.tile0) * kTileRows;
          for (int e = lane; e < kTileRows * MT; e += 32) {
            const int r = e / MT, m = e - r * MT;
            const float v = ((buf[e] + buf[kTileRows * MT + e]) + buf[2 * kTileRows * MT + e]) + buf[3 * kTileRows * MT + e];
            const int row = row0 + r;
            if (row < N && m < M) {
              float* yp = T.y + (size_t)m * T.ldy + row;
              const float val = kFactor * v;
              *yp = kc0 == 0 ? val : *yp + val;
            }
          }
        }
      }
    }
    seg_begin = seg_end;
  }
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
  const size_t ring = (size_t)kQuads * G::RING * (G::SLOT + 256 + 16) + (size_t)kQuads * 2 * 4 * kTileRows * MT * 4;
  const size_t budget = kSmemMax - ring - 1024;
  // per staged column: M bf16 values
  const size_t per_col = (size_t)M * 2;
  int kc = (int)(budget / per_col) / kStep * kStep;
  const int need = (max_K + kStep - 1) / kStep * kStep;
  if (kc > need) kc = need;
  // One chunk that holds the longest K whole need not be a whole number of steps
  // (chunks past the first start at multiples of the chunk, which must then be
  // whole steps): at M = 4, K = 13824 fits in 108 KB but 14 steps do not.
  if (kc < max_K && (size_t)max_K * per_col <= budget) kc = max_K;
  if (kc < kStep) return fail(QMV_ERR_UNSUPPORTED, "activation chunk does not fit shared memory for M=%d", M);
  b.kc = kc;
  const size_t smem = ring + (size_t)M * kc * 2;
  fill_magic_bf16<FMT>(b.magic);
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
