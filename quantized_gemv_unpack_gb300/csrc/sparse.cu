// Flagged sparse ternary ("Ternary Bonsai 2", sections 1.1, 1.3, 3.3, 3.4, 5.5):
// block_ternary weights in which tiles of 16 rows x 128 columns whose codes are
// all zero are flagged in a per-group tile bitmap and not stored, and all-zero
// blocks carry the scale 1.0. The host packer converts a dense packed ternary
// buffer; the matvec is the fp16-FMA kernel of gemv.cu walking each row group's
// stored tiles.
//
// Matvec. One persistent launch (one CTA of W warps per SM: 20 up to M = 4, 16
// above) over a table of matvecs; rows are cut into tiles of W warps x RPW rows. A warp owns RPW rows
// of one 16-row group (the whole group at RPW = 16, a half at RPW = 8, a quarter
// at RPW = 4, which M >= 5 uses to stay within 128 registers) and
// walks the group's records (up to 8 stored tiles each, its rows contiguous in
// the record): lane 0 copies the warp's rows of a record into a two-slot ring
// with one bulk copy, two records ahead; lane 8g + p decodes stored tile p of
// the record for row quad g, reading the tile's block index to find its
// activations and its 16 rows' scales. Decode, staging and reduction are those
// of the dense kernel (gemv_core.cuh). The activations of a matvec are staged
// once (K must fit shared memory in one piece: records may straddle any split).
#include <algorithm>
#include <cstring>
#include <vector>

#include "gemv_core.cuh"

namespace qmv {

namespace {

using namespace core;

constexpr int kMaxSparseTasks = QMV_MAX_BATCH;
// Decode warps per CTA: 20 up to M = 4 (the kernel then fits 102 registers and
// the extra warps hide latency), 16 above.
template <int MT>
struct SparseWarps {
  static constexpr int value = MT <= 4 ? 20 : 16;
};

// one matvec; the sections are located by byte offsets from the packed buffer
struct SparseTask {
  const unsigned char* w;
  const uint16_t* x;   // bf16 [M][ldx]
  float* y;            // [M][ldy]
  uint32_t off_start, off_block, off_codes, off_scales;
  int32_t N, K, ldx, ldy, tile0, T;  // T: stored tiles (bounds the tile starts)
};

struct SparseBatch {
  int32_t n_tasks, n_tiles, kc, rows_per_tile, n_ctas, pad0;
  int32_t cta_tile[kMaxCtas + 1];
  uint32_t magic[10];
  int* err;
  SparseTask t[kMaxSparseTasks];
};

__device__ __forceinline__ int find_sparse_task(const SparseBatch& b, int tile) {
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// A ring slot holds the warp's rows of one record, then the record's tile
// scales (16 rows x up to 8 tiles of fp16, 32 bytes a tile), both copied on the
// slot's barrier.
template <int RPW, int W>
struct SparseRing {
  using G = Geometry<QMV_TERNARY2, RPW>;
  static constexpr int SLOT = G::SLOT + 256;
  static constexpr int RING = W * kSlots * SLOT;
  static constexpr int BARS = W * kSlots * 8;
};

template <int MT, int RPW>
__global__ void __launch_bounds__(SparseWarps<MT>::value * 32, 1)
    sparse_kernel(const __grid_constant__ SparseBatch b) {
  constexpr int FMT = QMV_TERNARY2;
  constexpr int W = SparseWarps<MT>::value;
  using F = Fmt<FMT>;
  using G = Geometry<FMT, RPW>;
  using R = SparseRing<RPW, W>;
  constexpr int RQ = RPW / kGroups;
  constexpr int TILE_ROWS = W * RPW;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + R::RING);
  const int S = b.kc / kStep;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw + R::RING + R::BARS);
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

  if (lane == 0) {
    for (int i = 0; i < kSlots; ++i) mbar_init(&wfull[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // the warp's rows of a tile: group g, rows half*RPW .. +RPW of it; records r of the group
  auto rows_of = [&](const SparseTask& T, int tile, int& g, int& half, uint32_t& t0, int& cnt) {
    const int wrow0 = (tile - T.tile0) * TILE_ROWS + warp * RPW;
    g = wrow0 / 16;
    half = (wrow0 % 16) / RPW;
    const uint32_t* start = reinterpret_cast<const uint32_t*>(T.w + T.off_start);
    if (wrow0 >= (T.N + 15) / 16 * 16) {
      t0 = 0;
      cnt = 0;
    } else {
      t0 = __ldg(start + g);
      cnt = (int)(__ldg(start + g + 1) - t0);
      if (cnt < 0 || cnt > T.K / 128 || t0 + (uint32_t)cnt > (uint32_t)T.T) {
        atomicCAS(b.err, 0, (int)QMV_ERR_CORRUPT);
        cnt = 0;
      }
    }
  };

  // ---- producer side of this warp: the warp's rows of a record and the record's
  // scales, two records ahead
  int p_tile = tile_begin, p_ti = 0, p_r = 0, p_cnt = 0, p_g = 0, p_half = 0;
  uint32_t p_t0 = 0, n_issued = 0;
  auto settle = [&]() {  // move to the next tile with records
    while (p_tile < tile_end) {
      p_ti = find_sparse_task(b, p_tile);
      rows_of(b.t[p_ti], p_tile, p_g, p_half, p_t0, p_cnt);
      if (p_cnt > 0) return;
      ++p_tile;
    }
  };
  settle();
  auto issue_one = [&]() {
    if (p_tile >= tile_end) return;
    const SparseTask& T = b.t[p_ti];
    const int nbk = min(kBlocksPerStep, p_cnt - p_r * kBlocksPerStep);
    const uint32_t bytes = (uint32_t)(RPW * nbk * G::BLOCK_BYTES);
    const int slot = n_issued % kSlots;
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const size_t tt = (size_t)p_t0 + (size_t)p_r * kBlocksPerStep;  // the record's first stored tile
      mbar_arrive_expect_tx(&wfull[slot], bytes + 32u * nbk);
      const unsigned char* src = T.w + T.off_codes + tt * 16 * G::BLOCK_BYTES + (size_t)p_half * RPW * nbk * G::BLOCK_BYTES;
      bulk_g2s(wring + (size_t)slot * R::SLOT, src, bytes, &wfull[slot]);
      bulk_g2s(wring + (size_t)slot * R::SLOT + G::SLOT, T.w + T.off_scales + tt * 32, 32u * nbk, &wfull[slot]);
    }
    ++n_issued;
    if (++p_r * kBlocksPerStep >= p_cnt) {
      p_r = 0;
      ++p_tile;
      settle();
    }
  };
  for (int i = 0; i < kSlots; ++i) issue_one();

  // ===================== decode
  const int g = lane >> 3;
  const int p = lane & 7;
  const DecodeK dk = load_decode_k(b.magic);
  const uint16_t* staged_x = nullptr;
  int staged_K = -1;
  uint32_t it = 0;

  for (int tile = tile_begin; tile < tile_end; ++tile) {
    const int ti = find_sparse_task(b, tile);
    const SparseTask& T = b.t[ti];
    if (T.x != staged_x || T.K != staged_K) {
      stage_chunk<FMT, MT, W * 32>(Bf16Rows{T.x, T.ldx, 0}, T.K, S, xs, s_red, s_xscale, s_xinv);
      staged_x = T.x;
      staged_K = T.K;
    }
    int grp, half, cnt;
    uint32_t t0;
    rows_of(T, tile, grp, half, t0, cnt);
    const uint16_t* tblock = reinterpret_cast<const uint16_t*>(T.w + T.off_block);
    float accc[RQ][MT];
#pragma unroll
    for (int r = 0; r < RQ; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) accc[r][m] = 0.f;
    const int nrec = (cnt + kBlocksPerStep - 1) / kBlocksPerStep;
    // block index of this lane's tile in a record, loaded one record ahead
    auto tile_block = [&](int rec) {
      return rec < nrec && rec * kBlocksPerStep + p < cnt ? (int)__ldg(tblock + t0 + (uint32_t)(rec * kBlocksPerStep + p))
                                                          : 0;
    };
    int blk_next = tile_block(0);
    for (int rec = 0; rec < nrec; ++rec, ++it) {
      const int nbk = min(kBlocksPerStep, cnt - rec * kBlocksPerStep);
      const bool active = p < nbk;
      int blk = blk_next;
      blk_next = tile_block(rec + 1);
      if (active && blk >= T.K / 128) {
        atomicCAS(b.err, 0, (int)QMV_ERR_CORRUPT);
        blk = 0;
      }
      const int slot = it % kSlots;
      mbar_wait(&wfull[slot], (it / kSlots) & 1u, b.err);
      if (active) {
        const unsigned char* sb = wring + (size_t)slot * R::SLOT;
        // the rows' scales of stored tile p: entries p * 16 + row of the record's scales
        const unsigned short* srec = reinterpret_cast<const unsigned short*>(sb + G::SLOT);
        unsigned short sc[RQ];
#pragma unroll
        for (int r = 0; r < RQ; ++r) sc[r] = srec[p * 16 + half * RPW + r * kGroups + g];
        decode_step<FMT, MT, RQ>(sb + p * G::BLOCK_BYTES, nbk * G::BLOCK_BYTES, xs, S, blk / kBlocksPerStep, g,
                                 blk % kBlocksPerStep, dk, sc, accc);
      }
      __syncwarp();
      issue_one();
    }
    // ---- reduce the eight lanes of each row, write y
    const int row0 = grp * 16 + half * RPW;
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int row = row0 + r * kGroups + g;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = accc[r][m] * s_xinv[m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (p == 0 && row < T.N) T.y[(size_t)m * T.ldy + row] = 2.f * v;
      }
    }
  }
}

template <int MT, int RPW>
int launch_sparse_t(SparseBatch& b, cudaStream_t s) {
  using G = Geometry<QMV_TERNARY2, RPW>;
  constexpr int W = SparseWarps<MT>::value;
  constexpr int TILE_ROWS = W * RPW;
  constexpr size_t kSmemMax = 227 * 1024;
  int tiles = 0, max_K = 0;
  for (int i = 0; i < b.n_tasks; ++i) {
    b.t[i].tile0 = tiles;
    tiles += (b.t[i].N + TILE_ROWS - 1) / TILE_ROWS;
    max_K = std::max(max_K, (int)b.t[i].K);
  }
  b.n_tiles = tiles;
  b.rows_per_tile = TILE_ROWS;
  const size_t fixed = SparseRing<RPW, W>::RING + SparseRing<RPW, W>::BARS;
  const int kc = (max_K + kStep - 1) / kStep * kStep;
  const size_t smem = fixed + (size_t)MT * kc * 2;
  if (smem > kSmemMax - 1024)
    return fail(QMV_ERR_UNSUPPORTED, "sparse ternary: K=%d with M=%d does not fit shared memory in one piece", max_K, MT);
  b.kc = kc;
  fill_magic<QMV_TERNARY2>(b.magic);
  b.err = device_error_word();
  if (!b.err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  auto kern = sparse_kernel<MT, RPW>;
  int per_sm = 0;
  int rc = kernel_fit((const void*)kern, W * 32, smem, &per_sm);
  if (rc) return rc;
  // persistent grid, one CTA per SM; contiguous tile ranges of about equal work,
  // a tile weighing rows x K x the matrix's stored fraction of 16 x 128 tiles
  const int grid = std::min(std::min(sm_count(), kMaxCtas), tiles);
  b.n_ctas = grid;
  std::vector<double> w(b.n_tasks);
  double total = 0;
  for (int i = 0; i < b.n_tasks; ++i) {
    const double groups = (double)((b.t[i].N + 15) / 16), blocks = (double)(b.t[i].K / 128);
    w[i] = (double)b.t[i].K * ((double)b.t[i].T / (groups * blocks));
    total += w[i] * b.t[i].N;
  }
  b.cta_tile[0] = 0;
  int c = 1;
  double done = 0;
  for (int i = 0; i < b.n_tasks && c < grid; ++i) {
    const int nt = (b.t[i].N + TILE_ROWS - 1) / TILE_ROWS;
    for (int j = 0; j < nt && c < grid; ++j) {
      done += w[i] * std::min(TILE_ROWS, (int)b.t[i].N - j * TILE_ROWS);
      while (c < grid && done >= total * c / grid) b.cta_tile[c++] = b.t[i].tile0 + j + 1;
    }
  }
  for (; c <= grid; ++c) b.cta_tile[c] = tiles;
  kern<<<grid, W * 32, smem, s>>>(b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse ternary launch");
  return QMV_OK;
}

int launch_sparse(SparseBatch& b, int M, cudaStream_t s) {
  switch (M) {
    case 1: return launch_sparse_t<1, 16>(b, s);
    case 2: return launch_sparse_t<2, 8>(b, s);
    case 3: return launch_sparse_t<3, 8>(b, s);
    case 4: return launch_sparse_t<4, 8>(b, s);
    case 5: return launch_sparse_t<5, 4>(b, s);
    case 6: return launch_sparse_t<6, 4>(b, s);
    case 7: return launch_sparse_t<7, 4>(b, s);
    case 8: return launch_sparse_t<8, 4>(b, s);
    default: return fail(QMV_ERR_ARG, "sparse ternary: M=%d outside 1..8", M);
  }
}

int64_t align256(int64_t n) { return (n + 255) / 256 * 256; }

void sparse_sections(int64_t N, int64_t K, int64_t T, int64_t* off, int64_t* bytes, int64_t* total) {
  const int64_t G = (N + 15) / 16, KB = K / 128;
  const int64_t sizes[5] = {G * ((KB + 31) / 32) * 4, (G + 1) * 4, T * 2, T * 16 * 32, T * 32};
  int64_t pos = 0;
  for (int i = 0; i < 5; ++i) {
    off[i] = pos;
    bytes[i] = sizes[i];
    pos = align256(pos + sizes[i]);
  }
  *total = pos;
}

}  // namespace

int check_sparse_desc(const qmv_desc* d) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  if (d->abi_version != QMV_ABI_VERSION || d->format != QMV_TERNARY2_SPARSE) return fail(QMV_ERR_ARG, "not a sparse ternary descriptor");
  if (d->N <= 0 || d->K <= 0 || d->K % 128 || d->group != 128) return fail(QMV_ERR_ARG, "N=%lld K=%lld group=%d", (long long)d->N, (long long)d->K, d->group);
  if (d->N > INT32_MAX / 2 || d->K > (1 << 26)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  const int64_t G = (d->N + 15) / 16, KB = d->K / 128;
  if (d->n_symbols < 0 || d->n_symbols > G * KB) return fail(QMV_ERR_ARG, "stored tiles %d outside 0..%lld", d->n_symbols, (long long)(G * KB));
  int64_t off[5], bytes[5], total;
  sparse_sections(d->N, d->K, d->n_symbols, off, bytes, &total);
  for (int i = 0; i < 5; ++i)
    if (off[i] != d->off[i] || bytes[i] != d->bytes[i]) return fail(QMV_ERR_ARG, "sparse ternary section %d does not match", i);
  if (total > (int64_t)UINT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "sparse ternary buffer above 4 GB");
  return QMV_OK;
}

// Run n sparse matvecs (descs already checked) with M activation rows in one launch.
int run_sparse(const qmv_desc* const* descs, const void* const* ws, const void* const* xs, const int64_t* ldx,
               float* const* ys, const int64_t* ldy, int n, int M, cudaStream_t s) {
  static thread_local SparseBatch b;
  if (n < 1 || n > kMaxSparseTasks) return fail(QMV_ERR_ARG, "n_tasks=%d outside 1..%d", n, kMaxSparseTasks);
  for (int i = 0; i < n; ++i) {
    const qmv_desc* d = descs[i];
    SparseTask& t = b.t[i];
    t.w = static_cast<const unsigned char*>(ws[i]);
    t.x = static_cast<const uint16_t*>(xs[i]);
    t.y = ys[i];
    t.off_start = (uint32_t)d->off[1];
    t.off_block = (uint32_t)d->off[2];
    t.off_codes = (uint32_t)d->off[3];
    t.off_scales = (uint32_t)d->off[4];
    t.N = (int32_t)d->N;
    t.K = (int32_t)d->K;
    t.ldx = (int32_t)ldx[i];
    t.ldy = (int32_t)ldy[i];
    t.tile0 = 0;
    t.T = d->n_symbols;
  }
  b.n_tasks = n;
  return launch_sparse(b, M, s);
}

}  // namespace qmv

using namespace qmv;

extern "C" {

int qmv_sparse_pack_host(const qmv_desc* dense, const void* dense_packed, qmv_desc* desc, void* out,
                         int64_t out_capacity) {
  int rc = check_desc(dense, QMV_TERNARY2);
  if (rc) return rc;
  if (!dense_packed || !desc) return fail(QMV_ERR_ARG, "NULL dense_packed or desc");
  const int64_t N = dense->N, K = dense->K, KB = K / 128, G = (N + 15) / 16, S = scale_steps(K);
  const unsigned char* base = static_cast<const unsigned char*>(dense_packed);
  const uint32_t* codes = reinterpret_cast<const uint32_t*>(base + dense->off[0]);
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(base + dense->off[1]);
  // word offset of (row r of group g, block b) in the dense record layout
  auto block_words = [&](int64_t g2, int64_t r, int64_t b2) {
    const int64_t st = b2 / 8, nbk = std::min<int64_t>(8, KB - st * 8);
    return codes + g2 * 16 * (K / 16) + st * 16 * 64 + r * nbk * 8 + (b2 % 8) * 8;
  };
  auto zero8 = [](const uint32_t* p) {
    uint32_t o = 0;
    for (int i = 0; i < 8; ++i) o |= p[i];
    return o == 0;
  };
  std::vector<int32_t> blocks;
  std::vector<uint32_t> start((size_t)G + 1, 0);
  for (int64_t g2 = 0; g2 < G; ++g2) {
    for (int64_t b2 = 0; b2 < KB; ++b2) {
      bool zero = true;
      for (int64_t r = 0; r < 16 && zero; ++r) zero = zero8(block_words(g2, r, b2));
      if (!zero) blocks.push_back((int32_t)b2);
    }
    start[g2 + 1] = (uint32_t)blocks.size();
  }
  const int64_t T = (int64_t)blocks.size();
  memset(desc, 0, sizeof(*desc));
  desc->abi_version = QMV_ABI_VERSION;
  desc->format = QMV_TERNARY2_SPARSE;
  desc->N = N;
  desc->K = K;
  desc->group = 128;
  desc->n_symbols = (int32_t)T;
  sparse_sections(N, K, T, desc->off, desc->bytes, &desc->total_bytes);
  if (!out) return QMV_OK;
  if (out_capacity < desc->total_bytes) return fail(QMV_ERR_ARG, "out_capacity %lld < %lld", (long long)out_capacity, (long long)desc->total_bytes);
  unsigned char* o = static_cast<unsigned char*>(out);
  memset(o, 0, (size_t)desc->total_bytes);
  uint32_t* tilemap = reinterpret_cast<uint32_t*>(o + desc->off[0]);
  memcpy(o + desc->off[1], start.data(), (size_t)(G + 1) * 4);
  uint16_t* tblock = reinterpret_cast<uint16_t*>(o + desc->off[2]);
  uint32_t* ocodes = reinterpret_cast<uint32_t*>(o + desc->off[3]);
  uint16_t* oscales = reinterpret_cast<uint16_t*>(o + desc->off[4]);
  const int64_t KBw = (KB + 31) / 32;
  for (int64_t g2 = 0; g2 < G; ++g2) {
    const int64_t t0 = start[g2], cnt = start[g2 + 1] - t0;
    for (int64_t i = 0; i < cnt; ++i) {
      const int64_t b2 = blocks[t0 + i];
      tilemap[g2 * KBw + b2 / 32] |= 1u << (b2 % 32);
      tblock[t0 + i] = (uint16_t)b2;
      for (int64_t r = 0; r < 16; ++r) {
        const int64_t n = g2 * 16 + r;
        uint16_t sc = 0;
        if (n < N) {  // an all-zero block of a real row stores the scale 1.0
          sc = zero8(block_words(g2, r, b2)) ? (uint16_t)0x3C00 : scales[scale_index(n, b2, S)];
        }
        oscales[(t0 + i) * 16 + r] = sc;
      }
    }
    for (int64_t r0 = 0; r0 < cnt; r0 += 8) {  // records of up to 8 stored tiles, row after row
      const int64_t nbk = std::min<int64_t>(8, cnt - r0);
      uint32_t* rec = ocodes + (t0 + r0) * 16 * 8;
      for (int64_t r = 0; r < 16; ++r)
        for (int64_t i = 0; i < nbk; ++i) memcpy(rec + (r * nbk + i) * 8, block_words(g2, r, blocks[t0 + r0 + i]), 32);
    }
  }
  return QMV_OK;
}

}  // extern "C"
