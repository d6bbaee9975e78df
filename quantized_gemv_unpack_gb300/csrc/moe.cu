// Mixture-of-experts decode over ternary SwiGLU experts ("Nemotron 3.5 Bolt",
// expert top-K routing): only the experts the router selects are read.
//
// Two launches on the caller's stream; g and u pass between them in the
// caller's workspace. Each CTA of both starts by routing in shared memory (the
// same inputs and code give every CTA the same result; moe_route.cuh): one warp
// per token takes the top-k of its E logits (equal logits: lower expert first)
// as k rounds of a warp maximum over keys each lane keeps sorted, softmax over
// the k selected logits in fp32; then one thread per (token, expert) pair finds
// its place in expert-then-token order, and each active expert is listed once
// (a slot).
//  1. gate|up: a persistent grid (one CTA per SM) splits the units (slot,
//     tile of 80 rows of the [gate; up] matrix) into equal contiguous ranges;
//     a CTA stages the slot's token rows of x (gathered) once per slot and
//     decodes its rows with the same per-warp bulk-copy ring and decode step as
//     the matvec batch, prefetching across unit boundaries, and writes g and u
//     per (token, expert) pair to the workspace in fp32. The CTAs also zero y,
//     and CTA 0 leaves the routing (slots and pairs) in the workspace.
//  2. down: the same over the down matrices; staging computes h = silu(g) * u
//     (fp32) per pair, and the decoded rows are added into y[token] with
//     weight p by fp32 atomics (their order varies between runs; the sum stays
//     within the documented bound).
#include <algorithm>
#include <mutex>
#include <vector>

#include "gemv_core.cuh"
#include "lut.cuh"
#include "moe_route.cuh"

namespace qmv {
namespace {

using namespace core;

// Decode warps and rows per warp of the expert kernels, by the most tokens a
// slot can have (MT <= M): one token decodes 16 rows per warp (an activation
// load serves four rows, as in the matvec batch), two tokens 8, more tokens 4
// (4-row warps fit 102 registers at eight tokens, and 20 of them hide latency).
template <int MTMAX>
struct MoeCfg {
  static constexpr int W = MTMAX <= 2 ? 16 : 20;
  static constexpr int RPW = MTMAX == 1 ? 16 : (MTMAX == 2 ? 8 : 4);
  static constexpr int THREADS = W * 32;
  static constexpr int TILE_ROWS = W * RPW;
};
constexpr int kMoeSlots = 2;                            // ring slots per decode warp

// The expert kernels' ring: per warp kMoeSlots slots of one step of the warp's
// rows (a deeper ring measured slower at M = 1).
template <int W, int RPW>
struct MoeRing {
  using G = Geometry<QMV_TERNARY2, RPW>;
  static constexpr int SLOT = G::SLOT;
  static constexpr int RING = W * kMoeSlots * SLOT;
  static constexpr int BARS = W * kMoeSlots * 8;
};

// Workspace layout (all offsets in bytes from the workspace base).
struct MoeLayout {
  int64_t hdr, slot_expert, slot_first, slot_count, pair_token, pair_prob, gu, total;
  MoeLayout(int E, int topk, int M, int64_t I) {
    const int P = M * topk;
    const int S = std::min(E, P);
    auto al = [](int64_t v) { return (v + 255) / 256 * 256; };
    hdr = 0;
    slot_expert = al(hdr + 16);
    slot_first = al(slot_expert + 4 * S);
    slot_count = al(slot_first + 4 * S);
    pair_token = al(slot_count + 4 * S);
    pair_prob = al(pair_token + 4 * P);
    gu = al(pair_prob + 4 * P);
    total = al(gu + (int64_t)P * 2 * I * 4);
  }
};

struct MoeArgs {
  const uint32_t* gu_codes;   // expert 0's [gate; up] codes; expert e at + e * stride_words
  const uint16_t* gu_scales;
  const uint32_t* dn_codes;
  const uint16_t* dn_scales;
  int64_t stride_words;       // expert record stride in 32-bit words
  int64_t stride_halves;      // the same stride in 16-bit units
  const float* logits;        // [M][E]
  const uint16_t* x;          // bf16 [M][ldx]
  float* y;                   // [M][ldy]
  unsigned char* ws;
  int E, topk, M, H, I, ldx, ldy, max_slots;
  int64_t off_slot_expert, off_slot_first, off_slot_count, off_pair_token, off_pair_prob, off_gu;
  uint32_t magic[10];
  int* err;
};

// activation sources of the two expert phases
struct GatherRows {  // x rows of the slot's tokens
  const uint16_t* x;
  int ldx;
  const int* tok;    // shared memory, MT entries
  __device__ __forceinline__ void load8(int m, int k, float v[8]) const {
    Bf16Rows{x + (size_t)tok[m] * ldx, 0, 0}.load8(0, k, v);
  }
};
struct SwiGlu {  // h = silu(g) * u from the workspace, pair rows [first + m]
  const float* gu;
  int I, first;
  __device__ __forceinline__ void load8(int m, int k, float v[8]) const {
    const float* gr = gu + (size_t)(first + m) * 2 * I + k;
    const float4 g0 = *reinterpret_cast<const float4*>(gr), g1 = *reinterpret_cast<const float4*>(gr + 4);
    const float4 u0 = *reinterpret_cast<const float4*>(gr + I), u1 = *reinterpret_cast<const float4*>(gr + I + 4);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = g[e] / (1.f + __expf(-g[e])) * u[e];
  }
};

// Per-warp producer over the CTA's sequence of (unit, step), unit = (slot,
// tile): lane 0 copies the warp's 4 rows of one step of the unit's expert
// matrix into the next ring slot (one bulk copy, completes on the slot's
// mbarrier), two steps ahead of the decode.
template <int W, int RPW>
struct UnitProducer {
  const uint32_t* codes0;   // expert 0's codes; expert e at + e * stride_words
  int64_t stride_words;
  const int* slot_expert;   // shared memory
  int N, K, tiles, u, u_end, s, nsteps, warp, lane;
  uint32_t n_issued;
  unsigned char* wring;
  uint64_t* wfull;
  __device__ __forceinline__ void issue() {
    using F = Fmt<QMV_TERNARY2>;
    using G = Geometry<QMV_TERNARY2, RPW>;
    constexpr int kStepWords = kBlocksPerStep * F::WPB;
    if (u >= u_end) return;
    const int nb = K / 128;
    const int nbk = min(kBlocksPerStep, nb - s * kBlocksPerStep);
    const int wrow0 = (u % tiles) * (W * RPW) + warp * RPW;
    const int N16 = (N + 15) / 16 * 16;
    const uint32_t bytes = wrow0 < N16 ? (uint32_t)(RPW * nbk * G::BLOCK_BYTES) : 0u;
    const int slot = n_issued % kMoeSlots;
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&wfull[slot], bytes);
      if (bytes) {
        const uint32_t* codes = codes0 + (size_t)slot_expert[u / tiles] * stride_words;
        const size_t off = (size_t)(wrow0 / 16) * 16 * (K / F::CPW) + (size_t)s * 16 * kStepWords +
                           (size_t)(wrow0 % 16) * nbk * F::WPB;
        bulk_g2s(wring + (size_t)slot * G::SLOT, codes + off, bytes, &wfull[slot]);
      }
    }
    ++n_issued;
    if (++s >= nsteps) {
      s = 0;
      ++u;
    }
  }
};

// Decode the units [u, u_end) of one slot (all tiles of one expert matrix for
// the slot's MT tokens); out(m, row, value) receives sum_k w_hat x.
template <int W, int RPW, int MT, class Src, class Out>
__device__ void run_slot(const uint16_t* scales, int N, int K, int tiles, int u, int u_end, const Src& src,
                         const Out& out, unsigned char* smem_raw, const DecodeK& dk, UnitProducer<W, RPW>& prod,
                         uint32_t& it, int* err, bool restage) {
  constexpr int FMT = QMV_TERNARY2;
  using F = Fmt<FMT>;
  using G = Geometry<FMT, RPW>;
  using Ring = MoeRing<W, RPW>;
  constexpr int RQ = RPW / kGroups;
  __shared__ float s_red[W][MT];
  __shared__ float s_xinv[MT];
  __shared__ float s_xscale[MT];
  const int S = (K + kStep - 1) / kStep;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw + Ring::RING + Ring::BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 3, p = lane & 7;
  const int nb = K / 128;
  const int nsteps = (nb + kBlocksPerStep - 1) / kBlocksPerStep;
  const int KB = K / 128;

  if (restage) stage_chunk<FMT, MT, W * 32>(src, K, S, xs, s_red, s_xscale, s_xinv);

  const int SS = (KB + kBlocksPerStep - 1) / kBlocksPerStep;  // scale records per 16-row group
  for (; u < u_end; ++u) {
    const int wrow0 = (u % tiles) * (W * RPW) + warp * RPW;
    const unsigned short* sp[RQ];
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int row = min(wrow0 + r * kGroups + g, N - 1);
      sp[r] = reinterpret_cast<const unsigned short*>(scales) + (size_t)(row / 16) * SS * 128 +
              (row % 16) * kBlocksPerStep + p;
    }
    float accc[RQ][MT];
#pragma unroll
    for (int r = 0; r < RQ; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) accc[r][m] = 0.f;
    // block scales run one step ahead of the decode (their load latency overlaps a step)
    unsigned short scn[RQ];
#pragma unroll
    for (int r = 0; r < RQ; ++r) scn[r] = p < nb ? __ldg(sp[r]) : (unsigned short)0;
    for (int s = 0; s < nsteps; ++s, ++it) {
      const bool active = s * kBlocksPerStep + p < nb;
      unsigned short sc[RQ];
#pragma unroll
      for (int r = 0; r < RQ; ++r) sc[r] = scn[r];
      if (s + 1 < nsteps) {
        const bool next = (s + 1) * kBlocksPerStep + p < nb;
#pragma unroll
        for (int r = 0; r < RQ; ++r) scn[r] = next ? __ldg(sp[r] + (s + 1) * 128) : (unsigned short)0;
      }
      const int slot = it % kMoeSlots;
      mbar_wait(&prod.wfull[slot], (it / kMoeSlots) & 1u, err);
      if (active) {
        const int row_bytes = min(kBlocksPerStep, nb - s * kBlocksPerStep) * G::BLOCK_BYTES;
        decode_step<FMT, MT, RQ>(prod.wring + (size_t)slot * G::SLOT + p * G::BLOCK_BYTES, row_bytes, xs, S,
                                 s, g, p, dk, sc, accc);
      }
      __syncwarp();
      prod.issue();
    }
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      const int row = wrow0 + r * kGroups + g;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = accc[r][m];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        if (p == 0 && row < N) out(m, row, 2.f * v * s_xinv[m]);
      }
    }
  }
}

struct GuOut {  // g|u of pair first + m
  float* gu;
  int I2, first;
  __device__ __forceinline__ void operator()(int m, int row, float v) const {
    gu[(size_t)(first + m) * I2 + row] = v;
  }
};
struct DownOut {  // y[token] += p * value
  float* y;
  int ldy;
  const int* tok;
  const float* prob;
  __device__ __forceinline__ void operator()(int m, int row, float v) const {
    atomicAdd(y + (size_t)tok[m] * ldy + row, prob[m] * v);
  }
};

// Persistent: CTA c takes the contiguous unit range [c*U/G, (c+1)*U/G) of the
// U = n_slots * tiles units of this phase (all units are the same size).
template <int PHASE, int MTMAX>
__global__ void __launch_bounds__(MoeCfg<MTMAX>::THREADS, 1) moe_expert_kernel(const MoeArgs a) {
  constexpr int W = MoeCfg<MTMAX>::W, RPW = MoeCfg<MTMAX>::RPW;
  using Ring = MoeRing<W, RPW>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ int s_tok[kMaxTokens];
  __shared__ float s_prob[kMaxTokens];
  __shared__ MoeRoute R;
  // the down launch may start on SMs this grid frees; it waits for this grid's
  // results (g, u and the zeroed y) before it reads them
  if (PHASE == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  route(MoeRouting{a.logits, a.E, a.topk, a.M}, R);
  if (PHASE == 0) {
    // y is accumulated by the down phase's atomics
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.M * a.H; i += gridDim.x * blockDim.x)
      a.y[(size_t)(i / a.H) * a.ldy + i % a.H] = 0.f;
    if (blockIdx.x == 0) {  // the routing, for inspection: slots and pairs in the workspace layout
      const int np = a.M * a.topk;
      for (int i = threadIdx.x; i < np; i += blockDim.x) {
        reinterpret_cast<int*>(a.ws + a.off_pair_token)[i] = R.pair_token[i];
        reinterpret_cast<float*>(a.ws + a.off_pair_prob)[i] = R.pair_prob[i];
      }
      for (int i = threadIdx.x; i < R.n_slots; i += blockDim.x) {
        reinterpret_cast<int*>(a.ws + a.off_slot_expert)[i] = R.slot_expert[i];
        reinterpret_cast<int*>(a.ws + a.off_slot_first)[i] = R.slot_first[i];
        reinterpret_cast<int*>(a.ws + a.off_slot_count)[i] = R.slot_count[i];
      }
      if (threadIdx.x == 0) *reinterpret_cast<int*>(a.ws) = R.n_slots;
    }
  }
  const int ns = R.n_slots;
  const int* slot_expert = R.slot_expert;
  const int* slot_first = R.slot_first;
  const int* slot_count = R.slot_count;
  const int N = PHASE == 0 ? 2 * a.I : a.H;
  const int K = PHASE == 0 ? a.H : a.I;
  const int tiles = (N + W * RPW - 1) / (W * RPW);
  const int total = ns * tiles;
  const int u_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int u_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  if (u_begin >= u_end) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  UnitProducer<W, RPW> prod;
  prod.codes0 = PHASE == 0 ? a.gu_codes : a.dn_codes;
  prod.stride_words = a.stride_words;
  prod.slot_expert = slot_expert;
  prod.N = N;
  prod.K = K;
  prod.tiles = tiles;
  prod.u = u_begin;
  prod.u_end = u_end;
  prod.s = 0;
  prod.nsteps = (K / 128 + kBlocksPerStep - 1) / kBlocksPerStep;
  prod.warp = warp;
  prod.lane = lane;
  prod.n_issued = 0;
  prod.wring = smem_raw + (size_t)warp * kMoeSlots * Ring::SLOT;
  prod.wfull = reinterpret_cast<uint64_t*>(smem_raw + Ring::RING) + warp * kMoeSlots;
  if (lane == 0) {
    for (int i = 0; i < kMoeSlots; ++i) mbar_init(&prod.wfull[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  for (int i = 0; i < kMoeSlots; ++i) prod.issue();
  // down: routing done and the first weight copies in flight; the gate|up grid's
  // g, u and zeroed y are complete and visible after this
  if (PHASE == 1) asm volatile("griddepcontrol.wait;" ::: "memory");

  const DecodeK dk = load_decode_k(a.magic);
  float* gu = reinterpret_cast<float*>(a.ws + a.off_gu);
  const uint16_t* scales0 = PHASE == 0 ? a.gu_scales : a.dn_scales;
  uint32_t it = 0;
  bool staged = false;  // gate|up at one token: every slot stages the same x, once
  for (int u = u_begin; u < u_end;) {
    const int slot = u / tiles;
    const int u_stop = min(u_end, (slot + 1) * tiles);
    const int e = slot_expert[slot];
    const int first = slot_first[slot];
    const int cnt = slot_count[slot];
    __syncthreads();  // the previous slot's token table is no longer read
    if (threadIdx.x < cnt) {
      s_tok[threadIdx.x] = R.pair_token[first + threadIdx.x];
      s_prob[threadIdx.x] = R.pair_prob[first + threadIdx.x];
    }
    __syncthreads();
    const uint16_t* scales = scales0 + (size_t)e * a.stride_halves;
    const bool restage = !(PHASE == 0 && a.M == 1 && staged);
    staged = true;
    if (PHASE == 0) {
      const GatherRows src{a.x, a.ldx, s_tok};
      const GuOut out{gu, 2 * a.I, first};
      switch (cnt) {
#define QMV_MOE_CASE(m)                                                                                          \
  case m:                                                                                                        \
    if (m <= MTMAX)                                                                                              \
      run_slot<W, RPW, (m <= MTMAX ? m : 1)>(scales, N, K, tiles, u, u_stop, src, out, smem_raw, dk, prod, it, \
                                             a.err, restage);                                                    \
    break;
        QMV_MOE_CASE(1) QMV_MOE_CASE(2) QMV_MOE_CASE(3) QMV_MOE_CASE(4)
        QMV_MOE_CASE(5) QMV_MOE_CASE(6) QMV_MOE_CASE(7) QMV_MOE_CASE(8)
        default: break;
      }
    } else {
      const SwiGlu src{gu, a.I, first};
      const DownOut out{a.y, a.ldy, s_tok, s_prob};
      switch (cnt) {
        QMV_MOE_CASE(1) QMV_MOE_CASE(2) QMV_MOE_CASE(3) QMV_MOE_CASE(4)
        QMV_MOE_CASE(5) QMV_MOE_CASE(6) QMV_MOE_CASE(7) QMV_MOE_CASE(8)
#undef QMV_MOE_CASE
        default: break;
      }
    }
    u = u_stop;
  }
}

template <int MTMAX>
size_t expert_smem(int64_t K) {
  using Ring = MoeRing<MoeCfg<MTMAX>::W, MoeCfg<MTMAX>::RPW>;
  const int64_t S = (K + kStep - 1) / kStep;
  return Ring::RING + Ring::BARS + (size_t)MTMAX * S * kStep * 2;
}

// The two expert launches for slots of at most MTMAX tokens (MTMAX >= M).
template <int MTMAX>
int launch_experts(const MoeArgs& a, int64_t H, int64_t I, cudaStream_t s) {
  using Cfg = MoeCfg<MTMAX>;
  const size_t smem_gu = expert_smem<MTMAX>(H), smem_dn = expert_smem<MTMAX>(I);
  int per_sm = 0;
  int rc = kernel_fit((const void*)moe_expert_kernel<0, MTMAX>, Cfg::THREADS, smem_gu, &per_sm);
  if (rc) return rc;
  rc = kernel_fit((const void*)moe_expert_kernel<1, MTMAX>, Cfg::THREADS, smem_dn, &per_sm);
  if (rc) return rc;
  // persistent grids: one CTA per SM, capped by the largest possible unit count
  const int units_gu = a.max_slots * (int)((2 * I + Cfg::TILE_ROWS - 1) / Cfg::TILE_ROWS);
  const int units_dn = a.max_slots * (int)((H + Cfg::TILE_ROWS - 1) / Cfg::TILE_ROWS);
  moe_expert_kernel<0, MTMAX><<<std::min(sm_count(), units_gu), Cfg::THREADS, smem_gu, s>>>(a);
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return cuda_fail(ce, "moe gate|up launch");
  // programmatic dependent launch: the down grid's routing and first weight
  // copies overlap the end of the gate|up grid
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)std::min(sm_count(), units_dn));
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = smem_dn;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ce = cudaLaunchKernelEx(&cfg, moe_expert_kernel<1, MTMAX>, a);
  if (ce != cudaSuccess) return cuda_fail(ce, "moe down launch");
  return QMV_OK;
}

// Scratch for moe_qmv_run_static: one fixed array per device, in the module's
// own global memory, for callers that cannot allocate device memory.
__device__ __align__(256) unsigned char g_moe_static_scratch[QMV_MOE_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
std::vector<void*> g_static_ptr;  // device address of the scratch, per device ordinal

// Device address of the scratch array on the current device (looked up once).
int static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_static_mu);
  if ((int)g_static_ptr.size() <= dev) g_static_ptr.resize(dev + 1, nullptr);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(MoE static scratch)");
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return QMV_OK;
}

}  // namespace
}  // namespace qmv

using namespace qmv;

extern "C" {

size_t moe_workspace_size(int E, int topk, int M, int64_t H, int64_t I) {
  (void)H;
  if (E < 1 || topk < 1 || M < 1 || I < 1) return 0;
  return (size_t)MoeLayout(E, topk, M, I).total;
}

int moe_qmv_run(const qmv_desc* gateup_desc, const qmv_desc* down_desc, const void* experts, int64_t expert_stride,
                int64_t down_off, int E, const float* logits, int topk, const void* x_bf16, int M, int64_t ldx,
                float* y, int64_t ldy, void* workspace, size_t ws_bytes, void* stream) {
  // experts in the byte-lookup layout run on the lookup kernel, in the record layout on the FMA kernels
  const bool lut = gateup_desc && gateup_desc->format == QMV_TERNARY2_LUT;
  int rc = lut ? check_lut_desc(gateup_desc) : check_desc(gateup_desc, QMV_TERNARY2);
  if (rc) return fail(rc, "gate|up descriptor: %s", qmv_last_error());
  rc = lut ? check_lut_desc(down_desc) : check_desc(down_desc, QMV_TERNARY2);
  if (rc) return fail(rc, "down descriptor: %s", qmv_last_error());
  const int64_t H = gateup_desc->K, I2 = gateup_desc->N;
  if (I2 % 2 || down_desc->N != H || down_desc->K != I2 / 2)
    return fail(QMV_ERR_ARG, "shapes: [gate; up] must be 2I x H and down H x I");
  const int64_t I = I2 / 2;
  if (I % 128) return fail(QMV_ERR_ARG, "I=%lld must be a multiple of 128", (long long)I);
  if (E < 1 || E > kMaxExperts || topk < 1 || topk > kMaxTopk || topk > E || M < 1 || M > kMaxTokens)
    return fail(QMV_ERR_ARG, "E=%d topk=%d M=%d outside 1..256, 1..8 (<= E), 1..8", E, topk, M);
  if (!experts || !logits || !x_bf16 || !y || !workspace) return fail(QMV_ERR_ARG, "NULL pointer");
  if (!aligned16(experts) || !aligned16(logits) || !aligned16(x_bf16) || !aligned16(y) || !aligned16(workspace))
    return fail(QMV_ERR_ALIGN, "buffers must be 16-byte aligned");
  if (expert_stride % 256 || down_off % 256 || down_off < gateup_desc->total_bytes ||
      down_off + down_desc->total_bytes > expert_stride)
    return fail(QMV_ERR_ARG, "expert record: stride and down_off must be multiples of 256 and hold both matrices");
  if (ldx < H || ldx % 8 || ldy < H) return fail(QMV_ERR_ARG, "ldx/ldy");
  if (H > INT32_MAX || ldx > INT32_MAX || ldy > INT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "sizes too large");
  const MoeLayout L(E, topk, M, I);
  if (ws_bytes < (size_t)L.total) return fail(QMV_ERR_ARG, "workspace %zu < %lld bytes", ws_bytes, (long long)L.total);
  if (lut) {
    if (!device_error_word()) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
    const unsigned char* base = static_cast<const unsigned char*>(experts);
    LutMoeCall c;
    c.gu_codes = base + gateup_desc->off[0];
    c.dn_codes = base + down_off + down_desc->off[0];
    c.stride = expert_stride;
    c.logits = logits;
    c.E = E;
    c.topk = topk;
    c.M = M;
    c.H = H;
    c.I = I;
    c.x = static_cast<const uint16_t*>(x_bf16);
    c.ldx = ldx;
    c.y = y;
    c.ldy = ldy;
    c.ws = static_cast<unsigned char*>(workspace);
    c.off_slot_expert = L.slot_expert;
    c.off_slot_first = L.slot_first;
    c.off_slot_count = L.slot_count;
    c.off_pair_token = L.pair_token;
    c.off_pair_prob = L.pair_prob;
    c.off_gu = L.gu;
    return run_lut_moe(c, static_cast<cudaStream_t>(stream));
  }
  const size_t need_gu = M == 1 ? expert_smem<1>(H) : (M == 2 ? expert_smem<2>(H) : expert_smem<8>(H));
  const size_t need_dn = M == 1 ? expert_smem<1>(I) : (M == 2 ? expert_smem<2>(I) : expert_smem<8>(I));
  if (std::max(need_gu, need_dn) > 227 * 1024 - 1024) return fail(QMV_ERR_UNSUPPORTED, "hidden size too large for one CTA");
  int* err = device_error_word();
  if (!err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");

  MoeArgs a;
  const char* base = static_cast<const char*>(experts);
  a.gu_codes = reinterpret_cast<const uint32_t*>(base + gateup_desc->off[0]);
  a.gu_scales = reinterpret_cast<const uint16_t*>(base + gateup_desc->off[1]);
  a.dn_codes = reinterpret_cast<const uint32_t*>(base + down_off + down_desc->off[0]);
  a.dn_scales = reinterpret_cast<const uint16_t*>(base + down_off + down_desc->off[1]);
  a.stride_words = expert_stride / 4;
  a.stride_halves = expert_stride / 2;
  a.logits = logits;
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.y = y;
  a.ws = static_cast<unsigned char*>(workspace);
  a.E = E;
  a.topk = topk;
  a.M = M;
  a.H = (int)H;
  a.I = (int)I;
  a.ldx = (int)ldx;
  a.ldy = (int)ldy;
  a.max_slots = std::min(E, M * topk);
  a.off_slot_expert = L.slot_expert;
  a.off_slot_first = L.slot_first;
  a.off_slot_count = L.slot_count;
  a.off_pair_token = L.pair_token;
  a.off_pair_prob = L.pair_prob;
  a.off_gu = L.gu;
  core::fill_magic<QMV_TERNARY2>(a.magic);
  a.err = err;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 1) return launch_experts<1>(a, H, I, s);
  if (M == 2) return launch_experts<2>(a, H, I, s);
  return launch_experts<8>(a, H, I, s);
}

int moe_qmv_run_static(const qmv_desc* gateup_desc, const qmv_desc* down_desc, const void* experts,
                       int64_t expert_stride, int64_t down_off, int E, const float* logits, int topk,
                       const void* x_bf16, int M, int64_t ldx, float* y, int64_t ldy, void* stream) {
  if (!gateup_desc) return fail(QMV_ERR_ARG, "gate|up descriptor is NULL");
  const size_t need = moe_workspace_size(E, topk, M, gateup_desc->K, gateup_desc->N / 2);
  if (need == 0) return fail(QMV_ERR_ARG, "E=%d topk=%d M=%d", E, topk, M);
  if (need > (size_t)QMV_MOE_STATIC_SCRATCH_BYTES)
    return fail(QMV_ERR_ARG, "this MoE call needs %zu bytes of scratch; the static scratch holds %zu (use moe_qmv_run "
                "with a caller workspace)", need, (size_t)QMV_MOE_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  int rc = static_scratch(&scratch);
  if (rc) return rc;
  return moe_qmv_run(gateup_desc, down_desc, experts, expert_stride, down_off, E, logits, topk, x_bf16, M, ldx, y,
                     ldy, scratch, (size_t)QMV_MOE_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
