// Fused dequantize-and-matvec for block-128 ternary and group-128 INT4 weights.
//
// One persistent launch (one CTA per SM) walks a table of matvecs: one GEMV,
// the q|k|v group of a layer, or a whole decode stack. Rows are cut into tiles
// of W * RPW rows; the host gives every CTA a contiguous range of tiles holding
// about the same number of bytes, so a CTA re-stages its activations only when
// its range crosses into the next matvec. W = 16 decode warps per CTA; a launch
// too small to give every SM a 64-row tile uses 4-warp CTAs of 16 rows instead,
// several per SM.
//
// Streaming. Each warp owns RPW consecutive rows of
// the tile and a two-slot ring in shared memory; a slot holds one step (1024
// columns) of its rows. The packed codes are stored in records of 16 rows x
// one step, so a warp's rows of a step are one contiguous range: lane 0 of the
// warp fills a slot with a single 1D bulk copy (cp.async.bulk) that completes
// on the slot's mbarrier, two steps ahead of the step being decoded, walking
// the same (tile, chunk, step) sequence as the decode loop. Every wait gives
// up after 2 s and records QMV_ERR_TIMEOUT in the device error word instead of
// spinning on.
//
// Inside a decode warp, lane = 8*g + p: lane p (0..7) owns one 128-column
// block of the step and lane group g (0..3) one row of each row quad, so the
// warp decodes RPW rows x 1024 columns per step.
//
// Activations are staged per (x, chunk) in shared memory as fp16 pairs in
// the order a lane consumes them, after scaling the chunk by a power of two
// so its largest magnitude lies in [2^13, 2^14) (ternary) or [2^10, 2^11)
// (INT4); the scale is undone in fp32.
//
// Decode, per 32-bit code word, without lookup tables: one shift, one
// three-input logic op and one fp16 subtraction per column pair (mask and base
// live in registers). The ALU pipe (logic ops, shifts) and the FMA pipe
// (integer multiply, fp16 arithmetic) each issue 16 lanes per clock per SM
// sub-partition on this GPU, so of the eight ternary shifts per word four (the
// left shifts by 9, 7, 5, 1) are integer multiplies by 2^s and four are funnel
// shifts; the multipliers and amounts arrive as kernel parameters so the
// assembler keeps that split.
//  * ternary: the low half holds even columns, the high half odd columns, so a
//    word gives eight (even, odd) column pairs. Shifting pair i's two 2-bit
//    codes to bits 9-10 and 25-26 and computing (t & 0x06000600) ^ 0x3C003C00
//    yields two fp16 values v = 1 + q/2 (code 00 -> 1.0, 01 -> 1.5, 10 -> 0.5):
//    bit 9 is the mantissa MSB (+0.5), bit 10 the exponent LSB (halves 1.0).
//    Subtracting 1 gives q/2 exactly, so a zero code contributes exactly 0
//    whatever its activation; the factor 2 is applied at the end.
//  * INT4: (t & 0x000F000F) ^ 0x64086408 maps a two's-complement nibble q to
//    the fp16 integer 1032 + q (1024 + offset-binary nibble); subtracting 1032
//    gives q exactly.
// Products of these weights with the staged activations are exact. They are
// summed in fp16 chains of four column pairs, and each chain is widened into
// an fp32 block sum (two mixed-precision adds); the block sum is scaled by the
// block's fp16 scale in fp32. A chain rounds three times, so each row stays
// within 3 * 2^-11 (1.5e-3) of sum_k |w_hat_k x_k| plus fp32 rounding. Three
// warp shuffles reduce the eight lanes of a row at the end of the tile.
#include <algorithm>
#include <cstdlib>

#include "gemv_core.cuh"

namespace qmv {
namespace {

using namespace core;

__device__ __forceinline__ int find_task(const GemvBatch& b, int tile) {
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}


// A ring slot holds the warp's rows of one step, then the step's 256-byte
// scale record (16 rows x 8 blocks of fp16), both copied on the slot's barrier.
// W decode warps per CTA: 16 (one persistent CTA per SM) or, for launches too
// small to give every SM a 64-row tile, 4 (16-row tiles, several CTAs per SM).
template <int FMT, int RPW, int W>
struct FmaRing {
  using G = Geometry<FMT, RPW>;
  static constexpr int SLOT = G::SLOT + 256;
  static constexpr int RING = W * kSlots * SLOT;
  static constexpr int BARS = W * kSlots * 8;
  static constexpr int TILE_ROWS = W * RPW;
};

template <int FMT, int MT, int RPW, int W>
__global__ void __launch_bounds__(W * 32, 1) gemv_kernel(const __grid_constant__ GemvBatch b) {
  using F = Fmt<FMT>;
  using G = Geometry<FMT, RPW>;
  using R = FmaRing<FMT, RPW, W>;
  constexpr int WPB = F::WPB;
  constexpr int RQ = RPW / kGroups;          // row quads per decode warp
  constexpr bool TERN = FMT == QMV_TERNARY2;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;                                             // [warp][slot][RPW rows of a step | scales]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + R::RING);          // [warp][slot]
  const int KC = b.kc;
  const int S = KC / kStep;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw + R::RING + R::BARS);        // [MT][S][WPB][JW][8]
  __shared__ float s_red[W][MT];
  __shared__ float s_xinv[MT];
  __shared__ float s_xscale[MT];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int tile_begin = b.cta_tile[blockIdx.x];
  const int tile_end = b.cta_tile[blockIdx.x + 1];
  unsigned char* wring = ring + (size_t)warp * kSlots * R::SLOT;
  uint64_t* wfull = full + warp * kSlots;

  if (b.test_wait_us && test_wait_times_out(b.err, b.test_wait_us)) return;
  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(&wfull[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---- producer side of this warp: copy the warp's rows of one step and the
  // step's scale record into a slot. The source of the next step is one record
  // further on, except at a chunk's last (possibly partial) step or a new tile,
  // where it is located from scratch.
  constexpr int kStepWords = kBlocksPerStep * WPB;
  int p_tile = tile_begin, p_ti = 0, p_kc0 = 0, p_s = 0, p_nb = 0, p_K = 0;
  const uint32_t* p_src = nullptr;
  const uint16_t* p_ssrc = nullptr;
  uint32_t p_bytes = 0;
  auto p_locate = [&]() {
    const GemvTask& T = b.t[p_ti];
    p_K = T.K;
    p_nb = min(KC, p_K - p_kc0) / 128;
    const int nbk = min(kBlocksPerStep, p_nb - p_s * kBlocksPerStep);
    const int blk0 = p_kc0 / 128 + p_s * kBlocksPerStep;
    const int wrow0 = (p_tile - T.tile0) * R::TILE_ROWS + warp * RPW;
    const int N16 = (T.N + 15) / 16 * 16;
    // the warp's RPW rows lie inside one 16-row group: one contiguous piece of
    // the (group, step) record; rows past the padded end are not copied
    p_bytes = wrow0 < N16 ? (uint32_t)(RPW * nbk * G::BLOCK_BYTES) : 0u;
    p_src = T.codes + (size_t)(wrow0 / 16) * 16 * (p_K / F::CPW) + (size_t)(blk0 / kBlocksPerStep) * 16 * kStepWords +
            (size_t)(wrow0 % 16) * nbk * WPB;
    p_ssrc = T.scales + ((size_t)(wrow0 / 16) * scale_steps(p_K) + blk0 / kBlocksPerStep) * 128;
  };
  if (p_tile < tile_end) {
    p_ti = find_task(b, p_tile);
    p_locate();
  }
  uint32_t n_issued = 0;
  auto issue_one = [&]() {
    if (p_tile >= tile_end) return;
    const int slot = n_issued % kSlots;
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of the slot precede the copy
      mbar_arrive_expect_tx(&wfull[slot], p_bytes ? p_bytes + 256u : 0u);
      if (p_bytes) {
        bulk_g2s(wring + (size_t)slot * R::SLOT, p_src, p_bytes, &wfull[slot]);
        bulk_g2s(wring + (size_t)slot * R::SLOT + G::SLOT, p_ssrc, 256u, &wfull[slot]);
      }
    }
    ++n_issued;
    if ((++p_s + 1) * kBlocksPerStep <= p_nb) {  // another full step of this chunk
      p_src += 16 * kStepWords;
      p_ssrc += 128;
    } else {
      if (p_s * kBlocksPerStep >= p_nb) {
        p_s = 0;
        p_kc0 += KC;
        if (p_kc0 >= p_K) {
          p_kc0 = 0;
          if (++p_tile < tile_end) p_ti = find_task(b, p_tile);
        }
      }
      if (p_tile < tile_end) p_locate();
    }
  };
  for (int i = 0; i < kSlots; ++i) issue_one();

  // ===================== decode warps
  const int g = lane >> 3;
  const int p = lane & 7;
  const DecodeK dk = load_decode_k(b.magic);
  const uint16_t* staged_x = nullptr;
  int staged_kc0 = -1;
  int staged_K = -1;
  uint32_t it = 0;

  for (int tile = tile_begin; tile < tile_end; ++tile) {
    const int ti = find_task(b, tile);
    const uint16_t* __restrict__ x = b.t[ti].x;
    float* __restrict__ y = b.t[ti].y;
    const int N = b.t[ti].N, K = b.t[ti].K, ldx = b.t[ti].ldx, ldy = b.t[ti].ldy;
    const int wrow0 = (tile - b.t[ti].tile0) * R::TILE_ROWS + warp * RPW;
    const int srow = wrow0 % 16 + g;  // this lane's first row in the scale record

    float acc[RQ][MT];
#pragma unroll
    for (int r = 0; r < RQ; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    for (int kc0 = 0; kc0 < K; kc0 += KC) {
      const int kcn = min(KC, K - kc0);
      const int nb = kcn / 128;

      if (x != staged_x || kc0 != staged_kc0 || K != staged_K) {
        // ---- stage the activations of this chunk
        stage_chunk<FMT, MT, W * 32>(Bf16Rows{x, ldx, kc0}, kcn, S, xs, s_red, s_xscale, s_xinv);
        staged_x = x;
        staged_kc0 = kc0;
        staged_K = K;
      }

      // ---- decode this warp's rows over the chunk, one ring slot per step
      float accc[RQ][MT];
#pragma unroll
      for (int r = 0; r < RQ; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) accc[r][m] = 0.f;
      const int nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;

      for (int s = 0; s < nsteps; ++s, ++it) {
        const int slot = it % kSlots;
        mbar_wait(&wfull[slot], (it / kSlots) & 1u, b.err);
        if (s * kBlocksPerStep + p < nb) {
          const unsigned char* sb = wring + (size_t)slot * R::SLOT;
          // scales of (row, block p): entry row * 8 + p of the step's record
          const unsigned short* srec = reinterpret_cast<const unsigned short*>(sb + G::SLOT);
          unsigned short sc[RQ];
#pragma unroll
          for (int r = 0; r < RQ; ++r) sc[r] = srec[(srow + r * kGroups) * kBlocksPerStep + p];
          // rows of the step are nbk blocks apart in the slot
          const int row_bytes = min(kBlocksPerStep, nb - s * kBlocksPerStep) * G::BLOCK_BYTES;
          decode_step<FMT, MT, RQ>(sb + p * G::BLOCK_BYTES, row_bytes, xs, S, s, g, p, dk, sc, accc);
        }
        __syncwarp();  // every lane is done with the slot before it is refilled
        issue_one();
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float xinv = s_xinv[m];
#pragma unroll
        for (int r = 0; r < RQ; ++r) acc[r][m] = fmaf(accc[r][m], xinv, acc[r][m]);
      }
    }

    // ---- reduce the eight lanes of each row, write y
    constexpr float kFactor = TERN ? 2.f : 1.f;
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int row = wrow0 + r * kGroups + g;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = acc[r][m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (p == 0 && row < N) y[(size_t)m * ldy + row] = kFactor * v;
      }
    }
  }
}

// rows per decode warp: large for one activation row, small when the launch is
// too small to give every SM a tile or when many activation rows need registers
template <int FMT>
int pick_rpw(int M, int64_t total_rows) {
  const int big = M == 1 ? (FMT == QMV_TERNARY2 ? 16 : 8) : (M == 2 ? 8 : 4);
  if (big > 4 && total_rows / ((int64_t)kConsumerWarps * big) < sm_count()) return 4;
  return big;
}

template <int FMT, int MT, int RPW, int W = kConsumerWarps>
int launch_t(GemvBatch& b, cudaStream_t s) {
  using F = Fmt<FMT>;
  using R = FmaRing<FMT, RPW, W>;
  constexpr size_t kSmemMax = 227 * 1024;
  // tiles, numbered across tasks
  int tiles = 0;
  int max_K = 0;
  for (int i = 0; i < b.n_tasks; ++i) {
    b.t[i].tile0 = tiles;
    tiles += (b.t[i].N + R::TILE_ROWS - 1) / R::TILE_ROWS;
    max_K = std::max(max_K, (int)b.t[i].K);
  }
  b.n_tiles = tiles;
  b.rows_per_tile = R::TILE_ROWS;
  // activation chunk: as much of K as fits next to the ring, in whole steps;
  // per staged column: MT fp16 values
  const size_t fixed = R::RING + R::BARS;
  const size_t budget = kSmemMax - fixed - 1024;
  int kc_cap = (int)(budget / ((size_t)MT * kStep * 2)) * kStep;
  int kc = ((max_K + kStep - 1) / kStep) * kStep;
  if (kc > kc_cap) kc = kc_cap;
  if (kc < kStep) return fail(QMV_ERR_UNSUPPORTED, "activation chunk does not fit shared memory for M=%d", MT);
  b.kc = kc;
  const size_t smem = fixed + (size_t)MT * kc * 2;
  fill_magic<FMT>(b.magic);
  b.err = device_error_word();
  if (!b.err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  auto kern = gemv_kernel<FMT, MT, RPW, W>;
  int per_sm = 0;
  int rc = kernel_fit((const void*)kern, W * 32, smem, &per_sm);
  if (rc != QMV_OK) return rc;
  // persistent grid (16-warp CTAs: one per SM; smaller CTAs: as many as fit);
  // contiguous tile ranges of about equal bytes
  const int grid = std::min(std::min(sm_count() * (W == kConsumerWarps ? 1 : per_sm), kMaxCtas), tiles);
  double total = 0;
  for (int i = 0; i < b.n_tasks; ++i) total += (double)b.t[i].N * b.t[i].K;
  b.n_ctas = grid;
  b.cta_tile[0] = 0;
  int c = 1;
  double done = 0;
  for (int i = 0; i < b.n_tasks && c < grid; ++i) {
    const int nt = (b.t[i].N + R::TILE_ROWS - 1) / R::TILE_ROWS;
    for (int j = 0; j < nt && c < grid; ++j) {
      done += (double)std::min(R::TILE_ROWS, (int)b.t[i].N - j * R::TILE_ROWS) * b.t[i].K;
      while (c < grid && done >= total * c / grid) b.cta_tile[c++] = b.t[i].tile0 + j + 1;
    }
  }
  for (; c <= grid; ++c) b.cta_tile[c] = tiles;
  kern<<<grid, W * 32, smem, s>>>(b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
  return QMV_OK;
}

template <int FMT>
int launch_fmt(GemvBatch& b, int M, cudaStream_t s) {
  int64_t rows = 0;
  for (int i = 0; i < b.n_tasks; ++i) rows += b.t[i].N;
  const int rpw = pick_rpw<FMT>(M, rows);
  // fewer 64-row tiles than SMs: 4-warp CTAs of 16 rows instead
  const bool small = rpw == 4 && rows / ((int64_t)kConsumerWarps * 4) < sm_count();
  constexpr int BIG1 = FMT == QMV_TERNARY2 ? 16 : 8;
  switch (M) {
    case 1:
      return small ? launch_t<FMT, 1, 4, 4>(b, s) : rpw == 4 ? launch_t<FMT, 1, 4>(b, s) : launch_t<FMT, 1, BIG1>(b, s);
    case 2:
      return small ? launch_t<FMT, 2, 4, 4>(b, s) : rpw == 4 ? launch_t<FMT, 2, 4>(b, s) : launch_t<FMT, 2, 8>(b, s);
    case 3: return launch_t<FMT, 3, 4>(b, s);
    case 4: return launch_t<FMT, 4, 4>(b, s);
    case 5: return launch_t<FMT, 5, 4>(b, s);
    case 6: return launch_t<FMT, 6, 4>(b, s);
    case 7: return launch_t<FMT, 7, 4>(b, s);
    case 8: return launch_t<FMT, 8, 4>(b, s);
    default: return fail(QMV_ERR_ARG, "M=%d outside 1..8 for one launch", M);
  }
}

}  // namespace

int launch_gemv(int format, GemvBatch& b, int M, cudaStream_t s) {
  if (format == QMV_TERNARY2) return launch_fmt<QMV_TERNARY2>(b, M, s);
  if (format == QMV_INT4) return launch_fmt<QMV_INT4>(b, M, s);
  return fail(QMV_ERR_UNSUPPORTED, "format %d has no matvec kernel", format);
}

}  // namespace qmv
