// Batch-1 matvec over block-128 ternary weights in the lookup layout
// (QMV_TERNARY2_LUT): y = W_hat x for one activation row, with W_hat = q * s,
// q in {-1, 0, +1} per weight ("Ternary Bonsai 2", section 1.2) and one fp16
// scale s per block of 128 columns; and the same for group-128 INT4 weights
// in their lookup layout (QMV_INT4_LUT, "GPT-5.4" section 3.2), below.
//
// Decode by table lookup. A code byte holds the codes of four consecutive
// columns (2 bits each), so it takes one of 81 valid values e. Per block of
// 128 columns the CTA builds, from x, the table
//     T[e][c] = sum_{i<4} q_i(e) * x[128 b + 4 c + i]     (c = 0..31 column groups)
// in fp32 in shared memory; then every row's block costs one lookup per byte:
// 32 lookups, added in pairs by packed fp32x2 adds, and one multiply by the
// block's scale. The table has a 256-byte row per e, of which the first 32
// four-byte slots hold T[e][0..31]. The packer rotates each row's 32 code bytes
// by n % 32 (position t holds column group (t + n) % 32), so the lane that owns
// row n reads position t at slot (lane + t) mod 32: at every t the 32 lanes of
// a warp read 32 distinct banks (no conflicts). One byte permute builds the
// address e*256 + 4*((lane + t) mod 32) from the code word and a register whose
// bytes hold the lane's wrapped offsets of four consecutive positions (lane
// offsets plus 16 per code word, masked to 0..124: no carries between bytes).
// Rows of invalid bytes (a code 11) are zeroed once per launch and never
// rebuilt, so such a byte contributes 0.
//
// Occupancy. A CTA is 8 warps with 72 KB of shared memory (the table and the
// cluster partial sums) and 80 registers per thread, so three CTAs share an
// SM: their per-block barriers and table builds fall at different times and
// the lookups of one CTA fill the shared-memory pipe while another builds. One
// slot per entry (rather than a second copy at slot c + 32 to avoid the wrap)
// halves the table stores, which share the L1 data path with the lookups.
//
// Work split. A unit is up to 1024 rows of one matvec (its task's rows) over all of
// its blocks (a cluster of C CTAs splits the blocks, each CTA a contiguous
// share; then each CTA adds a 1/C share of the unit's rows over the C partial
// sums, in rank order, through distributed shared memory, so that the cluster
// finishes together). The host assigns units to CTAs (clusters) largest first,
// each to the least loaded one, and passes the lists in the launch parameters;
// when all units cost the same the device takes them round robin itself (no
// list to read), and tasks of one shape find their unit's task by a division.
// In a small batch a task whose units cost more than twice the median unit
// takes units of half or a quarter the rows. Each of the 256 threads owns up to
// four rows of a unit (rows r0 + 256 j + tid); lane = row % 32.
//
// INT4 (lut_kernel<QMV_INT4_LUT, 0>): a code byte is one column pair (two
// nibbles), so a block's table has 256 rows of 64 pair slots, T[lo + 16 hi][p] =
// q(lo) x[2p] + q(hi) x[2p + 1] (both products exact in fp32), built by all
// 256 threads (a pair and 64 byte values each); a row's block is 64 lookups,
// its 64 bytes read as two halves of 32, each rotated by n % 32 like the ternary
// bytes, the second half's slots 128 bytes on. 64 + 64 bytes of codes per row
// item need 128 registers, so two CTAs share an SM.
//
// MoE experts (lut_kernel<1>, <2>): the same kernel runs the gate|up and the down
// phase of the MoE decode over experts in this layout ("Nemotron 3.5 Bolt",
// expert top-K routing). Every CTA routes the tokens in shared memory; task i is
// the i-th (token, expert) pair in expert order, whose codes are its expert's
// matrix, whose activations are its token's x (gate|up) or h = silu(g) * u of
// its own gate|up outputs (down), and whose output goes to the workspace
// (gate|up) or is added, times the pair's routing weight, into y by fp32
// atomics (down). Each phase takes the cluster size whose rounds of units over
// the resident clusters, times steps per unit plus two, are fewest. The down
// launch is a programmatic dependent of the gate|up launch: it routes and loads
// its first weights while gate|up runs, and waits for it before reading g and u.
//
// Streaming. The codes of (block, 32-row group) are 1 KB records, rows of a
// unit contiguous per block, so a thread's row is two coalesced 16-byte loads.
// Right after a row's lookups its registers are reloaded with the same row slot
// of the next step, and one thread asks the copy engine to prefetch the step
// after next into L2 (cp.async.bulk.prefetch), so those loads hit L2. At its
// start a CTA asks for its second step by one L2 line prefetch per thread: the
// copy engine, busy with every CTA's requests at once, would hold its one thread
// back. (Asking for all of a small launch's weights at the start queued the first
// steps' loads behind them: MoE M = 1 29.5 against 28.6 us.) No wait in this
// kernel spins: it synchronizes only with CTA and cluster barriers and the
// dependent-launch wait.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "lut.cuh"
#include "moe_route.cuh"

namespace qmv {
namespace {

constexpr int kThreadsL = 256;                   // three CTAs per SM
constexpr int kRpt = 4;                          // rows per thread and unit
constexpr int kUnitRowsMax = kThreadsL * kRpt;   // 1024
constexpr int kMaxUnitsL = 4096;
constexpr int kMaxWorkersL = 512;
constexpr int kTableBytes = 65536;
constexpr int kPartBytes = 2 * kRpt * kThreadsL * 4;  // two unit parities of partial sums
// the table and the partial sums: 72 KB, so three CTAs (80 registers per
// thread) share an SM and one's table build overlaps the others' lookups
constexpr size_t kSmemL = kTableBytes + kPartBytes;

// Geometry of the two lookup layouts: bytes of a (block, 32-row group) record,
// code bytes of a row's block (table lookups per row and block), uint4 pieces
// of a row's block.
template <int FMT>
struct LutFmt;
template <>
struct LutFmt<QMV_TERNARY2_LUT> {
  static constexpr int REC = 1024, NPOS = 32, PIECES = 2, MIN_CTAS = 3;
};
template <>
struct LutFmt<QMV_INT4_LUT> {
  static constexpr int REC = 2048, NPOS = 64, PIECES = 4, MIN_CTAS = 2;
};

struct LutTask {
  const unsigned char* codes;  // section 0; the scales follow at NG * KB * record bytes
  const uint16_t* x;           // bf16 [K]
  float* y;                    // fp32 [N]
  int32_t N, rows, KB, unit0;  // rows per unit of this task (set by the launch), KB blocks, first unit
};

// The MoE expert phases (lut_kernel<1> gate|up, lut_kernel<2> down): task i is
// the i-th (token, expert) pair of the routing each CTA computes, its codes are
// expert e's matrix at codes + e * stride, and its activations and outputs are
// found from the pair.
struct LutMoe {
  MoeRouting routing;          // logits [M][E], E, topk, M
  const uint16_t* x;           // bf16 [M][ldx]
  float* y;                    // fp32 [M][ldy]: zeroed by gate|up, added into by down
  float* gu;                   // workspace: g (rows 0..I-1) and u (I..2I-1) of pair i at i * 2I
  unsigned char* ws;           // workspace base: gate|up's CTA 0 leaves the routing there
  int64_t off_slot_expert, off_slot_first, off_slot_count, off_pair_token, off_pair_prob;
  int64_t stride;              // bytes between experts' records
  int32_t I, H, ldx, ldy;
};

struct LutBatch {
  int32_t n_tasks, n_units, n_workers;
  int32_t sched_n;             // 0: unit u goes to worker u % n_workers
  int32_t upt;                 // units per task when every task has the same N (task = unit / upt), else 0
  uint32_t smem_bytes;         // dynamic shared memory of the launch
  int* err;
  LutMoe moe;
  uint16_t sched_off[kMaxWorkersL + 1];
  uint16_t sched[kMaxUnitsL];
  LutTask t[kMaxTasks];
};
static_assert(sizeof(LutBatch) <= 32000, "launch parameters must stay below the 32 KB limit");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
template <int IMM>
__device__ __forceinline__ float lds_at(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(IMM));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void l2_prefetch_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}
// Predicated loads: when pred is false the destination keeps its old value (no branch).
__device__ __forceinline__ void ldg16_if(uint4& v, const uint4* p, bool pred) {
  asm("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "l"(p), "r"((int)pred));
}
__device__ __forceinline__ void ldg2_if(uint32_t& v, const uint16_t* p, bool pred) {
  asm("{\n\t.reg .pred q;\n\t.reg .b16 h;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.global.nc.b16 h, [%1];\n\t@q cvt.u32.u16 %0, h;\n\t}"
      : "+r"(v)
      : "l"(p), "r"((int)pred));
}
// two fp32 adds in one instruction: (a.lo + lo, a.hi + hi)
__device__ __forceinline__ uint64_t add2_f32(uint64_t a, float lo, float hi) {
  uint64_t v, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(v));
  return d;
}
__device__ __forceinline__ float sum2_f32(uint64_t a) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(a));
  return __uint_as_float(lo) + __uint_as_float(hi);
}
__device__ __forceinline__ float code_val(int d, float x) { return d == 1 ? x : (d == 2 ? -x : 0.f); }

// One step = one block of one unit for this CTA.
struct Step {
  int k;        // position in this worker's unit list (past the end: no step)
  int ti, r0;   // task, first row of the unit
  int bk, kb1;  // current block, end of this CTA's blocks
  int nrows;    // rows of the unit
  bool valid;
  __device__ __forceinline__ int nrows32() const { return (nrows + 31) & ~31; }
};

template <int PIECES>
struct Item {
  uint4 c[PIECES];  // the row's code bytes of the block (32 ternary, 64 INT4)
  uint32_t s;       // the row's fp16 scale of the block (low 16 bits)
};

__device__ __forceinline__ int find_lut_task(const LutBatch& b, int unit) {
  if (b.upt) return unit / b.upt;
  int lo = 0, hi = b.n_tasks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.t[mid].unit0 <= unit) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

// FMT: QMV_TERNARY2_LUT or QMV_INT4_LUT. PHASE 0: the tasks' matvecs; 1 / 2: the
// MoE gate|up / down phase (see LutMoe; ternary only).
template <int FMT, int PHASE>
__global__ void __launch_bounds__(kThreadsL, LutFmt<FMT>::MIN_CTAS) lut_kernel(const __grid_constant__ LutBatch b) {
  using LF = LutFmt<FMT>;
  using ItemT = Item<LF::PIECES>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // the down phase may start on SMs the gate|up grid frees; it waits for that
  // grid's g, u and zeroed y before reading them
  if (PHASE == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the table: 256 rows (code byte e) of 256 bytes (slots 0..31 used), then the partial sums
  const uint32_t T0 = smem_u32(smem_raw);
  if (b.smem_bytes < kSmemL) {  // a launch without room for both: report, compute nothing
    if (threadIdx.x == 0) atomicCAS(b.err, 0, (int)QMV_ERR_UNSUPPORTED);
    return;
  }
  const uint32_t part = T0 + kTableBytes;     // [2][kRpt][kThreadsL] fp32
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // byte j of L0: 4 lane + 4 j (at most 136, so adding 16 k to every byte never carries)
  const uint32_t L0 = (uint32_t)(4 * lane) * 0x01010101u + 0x0C080400u;
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int worker = (int)cluster_id();

  // MoE phases: the routing of the M tokens, in shared memory (every CTA gets the
  // same result), and the expert of each pair
  MoeRoute* R = nullptr;
  int* pair_expert = nullptr;
  if constexpr (PHASE > 0) {
    __shared__ MoeRoute s_route;
    R = &s_route;
    route(b.moe.routing, *R);
    pair_expert = R->pair_expert;
    if constexpr (PHASE == 1) {
      const LutMoe& mo = b.moe;
      for (int i = blockIdx.x * kThreadsL + tid; i < mo.routing.M * mo.H; i += gridDim.x * kThreadsL)
        mo.y[(size_t)(i / mo.H) * mo.ldy + i % mo.H] = 0.f;
      if (blockIdx.x == 0) {  // the routing, for inspection, in the workspace layout
        const int np = mo.routing.M * mo.routing.topk;
        for (int i = tid; i < np; i += kThreadsL) {
          reinterpret_cast<int*>(mo.ws + mo.off_pair_token)[i] = R->pair_token[i];
          reinterpret_cast<float*>(mo.ws + mo.off_pair_prob)[i] = R->pair_prob[i];
        }
        for (int i = tid; i < R->n_slots; i += kThreadsL) {
          reinterpret_cast<int*>(mo.ws + mo.off_slot_expert)[i] = R->slot_expert[i];
          reinterpret_cast<int*>(mo.ws + mo.off_slot_first)[i] = R->slot_first[i];
          reinterpret_cast<int*>(mo.ws + mo.off_slot_count)[i] = R->slot_count[i];
        }
        if (tid == 0) *reinterpret_cast<int*>(mo.ws) = R->n_slots;
      }
    }
    __syncthreads();
  }
  // the codes of task ti (MoE: of its pair's expert)
  auto codes_of = [&](int ti) -> const unsigned char* {
    if constexpr (PHASE == 0) return b.t[ti].codes;
    else return b.t[0].codes + (size_t)pair_expert[ti] * (size_t)b.moe.stride;  // one base for every pair
  };
  // rows, 32-row groups and blocks of task ti
  struct Geo {
    int N, NG, KB;
  };
  auto geo = [&](int ti) -> Geo {
    const LutTask& T = b.t[ti];
    return Geo{T.N, (T.N + 31) >> 5, T.KB};
  };

  // this worker's units
  int k_end, k_beg;
  if (b.sched_n) {
    k_beg = b.sched_off[worker];
    k_end = b.sched_off[worker + 1];
  } else {
    k_beg = 0;
    k_end = worker < b.n_units ? (b.n_units - 1 - worker) / b.n_workers + 1 : 0;
  }
  auto unit_at = [&](int k) { return b.sched_n ? (int)b.sched[k] : worker + k * b.n_workers; };
  // first step of the unit at list position k (valid = false past the end)
  auto unit_step = [&](int k) {
    Step s = {};  // every field defined, also past the end of the list
    s.k = k;
    s.valid = k < k_end;
    if (!s.valid) return s;
    const int unit = unit_at(k);
    s.ti = find_lut_task(b, unit);
    const LutTask& T = b.t[s.ti];
    s.r0 = (unit - T.unit0) * T.rows;
    s.nrows = min(T.rows, T.N - s.r0);
    s.bk = (int)(rank * (uint32_t)T.KB / C);
    s.kb1 = (int)((rank + 1) * (uint32_t)T.KB / C);
    return s;
  };
  auto advance = [&](Step s) {
    if (!s.valid) return s;
    if (++s.bk < s.kb1) return s;
    return unit_step(s.k + 1);
  };
  // one thread: ask the copy engine to bring a step's code records (contiguous)
  // and scales into L2; it issues no load of its own, so the lookups' L1 path
  // stays free, but it may wait while the engine is busy
  auto prefetch_step_bulk = [&](const Step& s) {
    if (!s.valid) return;
    const Geo T = geo(s.ti);
    const unsigned char* codes = codes_of(s.ti);
    const int g0 = s.r0 >> 5;
    const int ng = s.nrows32() >> 5;
    l2_prefetch_bulk(codes + ((size_t)s.bk * T.NG + g0) * LF::REC, (uint32_t)ng * LF::REC);
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(codes + (size_t)T.NG * T.KB * LF::REC);
    l2_prefetch_bulk(sc + (size_t)s.bk * T.NG * 32 + s.r0, (uint32_t)ng * 64u);
  };
  // all threads: the same by one 128-byte line per thread and pass (never waits)
  auto prefetch_step = [&](const Step& s) {
    if (!s.valid) return;
    const Geo T = geo(s.ti);
    const unsigned char* codes = codes_of(s.ti);
    const int g0 = s.r0 >> 5;
    const int ng = s.nrows32() >> 5;
    const unsigned char* c0 = codes + ((size_t)s.bk * T.NG + g0) * LF::REC;
    const uint32_t nc = (uint32_t)ng * LF::REC;
    for (uint32_t o = (uint32_t)tid * 128u; o < nc; o += kThreadsL * 128u) l2_prefetch_line(c0 + o);
    const unsigned char* s0 = codes + (size_t)T.NG * T.KB * LF::REC + ((size_t)s.bk * T.NG * 32 + s.r0) * 2;
    const uint32_t ns = (uint32_t)ng * 64u;
    if ((uint32_t)tid * 128u < ns + 128u) l2_prefetch_line(s0 + min((uint32_t)tid * 128u, ns - 1u));
  };
  // This thread's load addresses of a step: row r0 + tid of its codes and of
  // its scales; item j (row r0 + 256 j + tid) is 8 row groups further on (8 KB
  // of codes, 512 B of scales). n32 > 256 j while item j has rows of this warp.
  struct Src {
    const uint4* cw;
    const uint16_t* sc;
    int n32;
  };
  auto src_of = [&](const Step& s) {
    Src r;
    r.cw = nullptr;
    r.sc = nullptr;
    r.n32 = 0;
    if (!s.valid) return r;
    const Geo T = geo(s.ti);
    const unsigned char* codes = codes_of(s.ti);
    r.cw = reinterpret_cast<const uint4*>(codes) + ((size_t)s.bk * T.NG + (s.r0 >> 5) + (tid >> 5)) * (LF::REC / 16) +
           lane;
    r.sc = reinterpret_cast<const uint16_t*>(codes + (size_t)T.NG * T.KB * LF::REC) + (size_t)s.bk * T.NG * 32 + s.r0 +
           tid;
    r.n32 = s.nrows32() - (tid & ~31);
    return r;
  };
  // piece i of a row holds its bytes 16i .. 16i+15, 512 bytes after piece i - 1
  auto load_item = [&](const Src& r, int j, ItemT& it) {
    const bool on = j * kThreadsL < r.n32;
#pragma unroll
    for (int i = 0; i < LF::PIECES; ++i) ldg16_if(it.c[i], r.cw + j * (kThreadsL / 32) * (LF::REC / 16) + 32 * i, on);
    ldg2_if(it.s, r.sc + j * kThreadsL, on);
  };
  // table builders: thread (warp w, lane g) writes column group g's entries of
  // the code bytes whose high digit pair (d2, d3) is hi = w (w < 8, nine bytes),
  // and of hi = 8 the byte with low pair lo = w (warp 0 also lo = 8)
  const int g = lane, warp = tid >> 5;
  // activations 4g .. 4g+3 of a step's block (MoE down: h = silu(g) * u of the pair)
  auto load_x = [&](const Step& s) -> float4 {
    if (!s.valid) return make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (PHASE == 2) {
      const float* gr = b.moe.gu + (size_t)s.ti * 2 * b.moe.I + (size_t)s.bk * 128 + 4 * g;
      const float4 gg = *reinterpret_cast<const float4*>(gr);
      const float4 uu = *reinterpret_cast<const float4*>(gr + b.moe.I);
      return make_float4(silu(gg.x) * uu.x, silu(gg.y) * uu.y, silu(gg.z) * uu.z, silu(gg.w) * uu.w);
    } else if constexpr (FMT == QMV_INT4_LUT) {
      // columns 2p, 2p + 1 of the thread's pair p = lane + 32 (warp & 1)
      const uint32_t xw = *reinterpret_cast<const uint32_t*>(b.t[s.ti].x + (size_t)s.bk * 128 + 2 * (g + 32 * (warp & 1)));
      return make_float4(__uint_as_float(xw << 16), __uint_as_float(xw & 0xFFFF0000u), 0.f, 0.f);
    } else {
      const uint16_t* xr = PHASE == 0 ? b.t[s.ti].x : b.moe.x + (size_t)R->pair_token[s.ti] * b.moe.ldx;
      const uint2 xw = *reinterpret_cast<const uint2*>(xr + (size_t)s.bk * 128 + 4 * g);
      return make_float4(__uint_as_float(xw.x << 16), __uint_as_float(xw.x & 0xFFFF0000u),
                         __uint_as_float(xw.y << 16), __uint_as_float(xw.y & 0xFFFF0000u));
    }
  };

  float acc[kRpt];
#pragma unroll
  for (int j = 0; j < kRpt; ++j) acc[j] = 0.f;
  int parity = 0;

  // the table of a step's block, from its x, into the table at tb
  auto build = [&](float4 xv, uint32_t tb) {
    const float x0 = xv.x, x1 = xv.y, x2 = xv.z, x3 = xv.w;
    if constexpr (FMT == QMV_INT4_LUT) {
      // INT4: thread (warp w, lane) writes pair p = lane + 32 (w & 1) of the 64 code
      // bytes whose high nibble is one of 4 (w >> 1) .. 4 (w >> 1) + 3:
      // T[lo + 16 hi][p] = q(lo) x0 + q(hi) x1, q the 4-bit two's complement value;
      // both products are exact in fp32
      const uint32_t slot = 4u * (uint32_t)(g + 32 * (warp & 1));
      float a[16];
#pragma unroll
      for (int lo = 0; lo < 16; ++lo) a[lo] = (float)(lo < 8 ? lo : lo - 16) * x0;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int hi = 4 * (warp >> 1) + hh;
        const float bh = (float)(hi < 8 ? hi : hi - 16) * x1;
#pragma unroll
        for (int lo = 0; lo < 16; ++lo) sts_f32(tb + (uint32_t)((hi * 16 + lo) * 256) + slot, a[lo] + bh);
      }
      return;
    }
    auto put = [&](int d0, int d1, int d2, int d3, float p23) {
      const float v = (code_val(d0, x0) + code_val(d1, x1)) + p23;
      const uint32_t a = tb + (uint32_t)((d0 + 4 * d1 + 16 * d2 + 64 * d3) * 256 + 4 * g);
      sts_f32(a, v);
    };
    {
      const int d2 = warp % 3, d3 = warp / 3;
      const float p23 = code_val(d2, x2) + code_val(d3, x3);
#pragma unroll
      for (int lo = 0; lo < 9; ++lo) put(lo % 3, lo / 3, d2, d3, p23);
    }
    const float p23 = -x2 - x3;  // hi = 8: d2 = d3 = 2 (codes 10, -1)
    put(warp % 3, warp / 3, 2, 2, p23);
    if (warp == 0) put(2, 2, 2, 2, p23);
  };
  // one row's block: one lookup per code byte (32 ternary, 64 INT4) and the adds,
  // times the block's scale, into acc. Positions 32..63 (INT4) are the second half,
  // rotated like the first, whose table slots are 32..63 (128 bytes on).
  auto row_block = [&](const ItemT& it, float& a, uint32_t tb) {
    uint32_t w[4 * LF::PIECES];
#pragma unroll
    for (int i = 0; i < LF::PIECES; ++i) {
      w[4 * i] = it.c[i].x;
      w[4 * i + 1] = it.c[i].y;
      w[4 * i + 2] = it.c[i].z;
      w[4 * i + 3] = it.c[i].w;
    }
    uint64_t s2 = 0;  // two partial sums (even and odd positions)
#pragma unroll
    for (int t = 0; t < LF::NPOS; t += 2) {
      // result bytes: wrapped lane offset, code byte t, 0, 0; plus the table base
      const uint32_t j0 = (uint32_t)(t & 3), j1 = (uint32_t)((t + 1) & 3);
      // byte j of Lk: (4 lane + 4 (4k + j)) mod 128, the wrapped slot offset of position 4k + j
      const uint32_t Lk = (L0 + (uint32_t)((t >> 2) & 7) * 0x10101010u) & 0x7C7C7C7Cu;
      const uint32_t tbh = tb + (t >= 32 ? 128u : 0u);
      const uint32_t a0 = prmt(w[t >> 2], Lk, (4u + j0) | (j0 << 4) | ((12u + j0) << 8) | ((12u + j0) << 12)) + tbh;
      const uint32_t a1 = prmt(w[(t + 1) >> 2], Lk, (4u + j1) | (j1 << 4) | ((12u + j1) << 8) | ((12u + j1) << 12)) + tbh;
      const float v0 = lds_at<0>(a0);
      const float v1 = lds_at<0>(a1);
      s2 = add2_f32(s2, v0, v1);
    }
    a = fmaf(sum2_f32(s2), __half2float(__ushort_as_half((unsigned short)it.s)), a);
  };
  // this thread's rows of a step (all four in a full unit, else the rows of this
  // warp's 32-row groups that the unit has); right after a row's block, its
  // register slot is reloaded with the same slot of the next step
  auto lookups = [&](const Step& s, ItemT (&it)[kRpt], const Src& n, uint32_t tb) {
    if (s.nrows32() == kUnitRowsMax) {
#pragma unroll
      for (int j = 0; j < kRpt; ++j) {
        row_block(it[j], acc[j], tb);
        load_item(n, j, it[j]);
      }
    } else {
      const int n32 = s.nrows32() - (tid & ~31);
#pragma unroll
      for (int j = 0; j < kRpt; ++j) {
        if (j * kThreadsL < n32) row_block(it[j], acc[j], tb);
        load_item(n, j, it[j]);
      }
    }
  };
  // the unit of s is complete in this CTA: write y (C == 1) or add the
  // cluster's partial sums in rank order (rank 0 writes)
  auto store = [&](const Step& s, int row, float v) {
    if constexpr (PHASE == 0) b.t[s.ti].y[row] = v;
    else if constexpr (PHASE == 1) b.moe.gu[(size_t)s.ti * 2 * b.moe.I + row] = v;
    else atomicAdd(b.moe.y + (size_t)R->pair_token[s.ti] * b.moe.ldy + row, R->pair_prob[s.ti] * v);
  };
  auto finish = [&](const Step& s) {
    if (C == 1) {
#pragma unroll
      for (int j = 0; j < kRpt; ++j) {
        const int row = s.r0 + j * kThreadsL + tid;
        if (j * kThreadsL + tid < s.nrows) store(s, row, acc[j]);
      }
    } else {
      const uint32_t pbase = part + (uint32_t)(parity * kRpt * kThreadsL * 4);
#pragma unroll
      for (int j = 0; j < kRpt; ++j) sts_f32(pbase + (uint32_t)((j * kThreadsL + tid) * 4), acc[j]);
      cluster_sync();
      // CTA `rank` adds its share of the unit's rows over the C partial sums, in rank
      // order, and stores them (every CTA of the cluster reads every other one's sums)
      const int per = (s.nrows + (int)C - 1) / (int)C;
      const int u_end = min((int)(rank + 1) * per, s.nrows);
      for (int u = (int)rank * per + tid; u < u_end; u += kThreadsL) {
        const uint32_t a = pbase + (uint32_t)(u * 4);
        float v = 0.f;
        for (uint32_t r = 0; r < C; ++r) v += ld_cluster_f32(a, r);
        store(s, s.r0 + u, v);
      }
      parity ^= 1;
    }
#pragma unroll
    for (int j = 0; j < kRpt; ++j) acc[j] = 0.f;
  };

  // Per step: prefetch the step after next to L2 and load the next step's
  // activations (builders); between two CTA barriers build the table; then look
  // up this step's rows, each slot reloaded with the next step's row at once.
  Step cur = unit_step(k_beg);
  Step nxt = advance(cur);
  ItemT A[kRpt];
#pragma unroll
  for (int j = 0; j < kRpt; ++j) {
#pragma unroll
    for (int i = 0; i < LF::PIECES; ++i) A[j].c[i] = make_uint4(0u, 0u, 0u, 0u);
    A[j].s = 0u;
  }
  {
    const Src first = src_of(cur);
#pragma unroll
    for (int j = 0; j < kRpt; ++j) load_item(first, j, A[j]);
  }
  prefetch_step(nxt);
  // zero the table rows of invalid code bytes (any 2-bit field equal to 3) while
  // the first loads are in flight (the loop's first barrier orders the zeros
  // before any lookup)
  if constexpr (FMT == QMV_TERNARY2_LUT)
    for (int i = tid; i < 256 * 32; i += kThreadsL) {
      const int e = i >> 5;
      if ((e & (e >> 1)) & 0x55) sts_f32(T0 + (uint32_t)(e * 256 + 4 * (i & 31)), 0.f);
    }
  // MoE down: the weights above do not depend on the gate|up grid; g and u do
  if (PHASE == 2) asm volatile("griddepcontrol.wait;" ::: "memory");
  float4 xc = load_x(cur);
  while (cur.valid) {
    const Step nn = advance(nxt);
    if (tid == 0) prefetch_step_bulk(nn);
    const float4 xn = load_x(nxt);
    __syncthreads();  // every lookup of the previous step is done
    build(xc, T0);
    __syncthreads();  // the table is complete
    lookups(cur, A, src_of(nxt), T0);
    if (!nxt.valid || nxt.k != cur.k) finish(cur);
    cur = nxt;
    nxt = nn;
    xc = xn;
  }
  // no CTA leaves while a peer may still read its partial sums
  if (C > 1) cluster_sync();
}

}  // namespace

int check_lut_desc(const qmv_desc* d) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  if (d->abi_version != QMV_ABI_VERSION)
    return fail(QMV_ERR_ARG, "desc abi_version %u, library %d", d->abi_version, QMV_ABI_VERSION);
  if (d->format != QMV_TERNARY2_LUT && d->format != QMV_INT4_LUT)
    return fail(QMV_ERR_ARG, "desc format %u is not a lookup layout (QMV_TERNARY2_LUT, QMV_INT4_LUT)", d->format);
  if (d->N <= 0 || d->K <= 0 || d->group != QMV_GROUP || d->K % QMV_GROUP)
    return fail(QMV_ERR_ARG, "desc N=%lld K=%lld group=%d", (long long)d->N, (long long)d->K, d->group);
  if (d->N > (1 << 26) || d->K > (1 << 26)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
  qmv_desc ref;
  qmv_pack_desc((int)d->format, d->N, d->K, d->group, &ref);
  for (int i = 0; i < 2; ++i)
    if (ref.off[i] != d->off[i] || ref.bytes[i] != d->bytes[i])
      return fail(QMV_ERR_ARG, "desc section %d does not match the lookup layout of a %lld x %lld matrix", i,
                  (long long)d->N, (long long)d->K);
  return QMV_OK;
}

namespace {

// Clusters of c CTAs of a lookup kernel (72 KB of shared memory, 256 threads)
// that fit the device at once, looked up once per kernel, device and c.
int active_clusters(const void* kernel, int c, int* out) {
  struct Entry {
    const void* k;
    int dev, c, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.k == kernel && e.dev == dev && e.c == c) {
      *out = e.n;
      return QMV_OK;
    }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(c * 8));
  cfg.blockDim = dim3(kThreadsL);
  cfg.dynamicSmemBytes = kSmemL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nc = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&nc, kernel, &cfg);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
  if (nc < 1) return fail(QMV_ERR_UNSUPPORTED, "no cluster of %d CTAs fits the device", c);
  cache.push_back({kernel, dev, c, nc});
  *out = nc;
  return QMV_OK;
}

// Units, clusters and the schedule of the n tasks in b.t, then the launch of
// lut_kernel<PHASE> (as a programmatic dependent of the previous launch on the
// stream when pdl is set).
template <int FMT, int PHASE>
int launch_lut(LutBatch& b, int n, int min_kb, cudaStream_t s, bool pdl) {
  b.n_tasks = n;
  const int sms = sm_count();
  auto units_for = [&](int rows) {
    int64_t u = 0;
    for (int i = 0; i < n; ++i) u += (b.t[i].N + rows - 1) / rows;
    return u;
  };
  auto kernel = lut_kernel<FMT, PHASE>;
  int per_sm = 0;
  int rc = kernel_fit((const void*)kernel, kThreadsL, kSmemL, &per_sm);
  if (rc) return rc;
  // CTAs (c = 1) or clusters of c CTAs resident at once
  auto workers_for = [&](int c, int* w) -> int {
    if (c == 1) {
      *w = sms * per_sm;
      return QMV_OK;
    }
    return active_clusters((const void*)kernel, c, w);
  };
  // Rows per unit and CTAs per cluster (matvec batches): whole 1024-row units on
  // single CTAs when there are enough of them; otherwise smaller units whose
  // blocks a cluster of up to 8 CTAs shares, until the launch covers twice the SMs
  // (the INT4 layer set 74 -> 46 us, the 4096 x 4096 ternary matrix 13.2 -> 12.0 us
  // against covering them once). A schedule-length model (units of 512 rows for the
  // INT4 layer set) measured slower: 49.9 against 45.5 us.
  const int64_t target = 2 * (int64_t)sms;
  int rows = kUnitRowsMax, C = 1;
  if (PHASE > 0) {
    // MoE phases (1024-row units of equal cost): the cluster size whose rounds of
    // units (units over resident clusters) times steps per unit, plus two for the
    // fill and the reduction, are fewest; ties to the larger cluster. Against
    // covering the SMs once: M = 3 63.7 -> 52 us, M = 8 121.2 -> 107 us (graph-replayed),
    // M = 1, 2, 4 unchanged.
    const int64_t units = units_for(kUnitRowsMax);
    int64_t best = INT64_MAX;
    for (int c = 1; c <= 8 && c <= min_kb; c *= 2) {
      int w = 0;
      rc = workers_for(c, &w);
      if (rc) return rc;
      const int64_t t = (units + w - 1) / w * ((min_kb + c - 1) / c + 2);
      if (t <= best) best = t, C = c;
    }
  } else if (units_for(kUnitRowsMax) < 2 * (int64_t)sms) {
    bool done = false;
    for (int r : {kUnitRowsMax, 512, 256}) {
      for (int c = 1; c <= 8 && c <= min_kb; c *= 2) {
        rows = r;
        C = c;
        if (units_for(r) * c >= target) {
          done = true;
          break;
        }
      }
      if (done) break;
    }
  }
  // In a small launch, a task whose units cost more than twice the typical unit
  // (rows x blocks, the median over units) takes units of half or a quarter the
  // rows, so that its few long units do not set the launch's length (the INT4
  // layer set's down projection, K = 13824 against 5120).
  for (int i = 0; i < n; ++i) b.t[i].rows = rows;
  if (units_for(kUnitRowsMax) < 2 * (int64_t)sms && n > 1) {
    std::vector<std::pair<int64_t, int64_t>> uc;  // (unit cost, units)
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
      const int64_t nu = (b.t[i].N + rows - 1) / rows;
      uc.push_back({(int64_t)rows * b.t[i].KB, nu});
      total += nu;
    }
    std::sort(uc.begin(), uc.end());
    int64_t acc = 0, median = uc.back().first;
    for (const auto& p : uc)
      if ((acc += p.second) * 2 >= total) {
        median = p.first;
        break;
      }
    for (int i = 0; i < n; ++i)
      while (b.t[i].rows > 256 && (int64_t)b.t[i].rows * b.t[i].KB > 2 * median) b.t[i].rows /= 2;
  }
  int64_t n_units = 0;
  bool same_n = true, same_cost = true;
  for (int i = 0; i < n; ++i) {
    b.t[i].unit0 = (int32_t)n_units;
    n_units += (b.t[i].N + b.t[i].rows - 1) / b.t[i].rows;
    same_n = same_n && b.t[i].N == b.t[0].N;
    same_n = same_n && b.t[i].rows == b.t[0].rows;
    same_cost = same_cost && b.t[i].KB == b.t[0].KB && (b.t[i].N % b.t[i].rows == 0 || b.t[i].N < b.t[i].rows);
  }
  // tasks of one shape: the device finds a unit's task by a division (no search)
  b.upt = same_n ? (b.t[0].N + b.t[0].rows - 1) / b.t[0].rows : 0;
  // units of one cost: the greedy schedule below is the round robin, which the
  // device computes itself (no list to read)
  same_cost = same_cost && (same_n || n == 1);
  if (n_units > INT32_MAX / 2) return fail(QMV_ERR_UNSUPPORTED, "batch too large");
  b.n_units = (int32_t)n_units;
  b.err = device_error_word();
  if (!b.err) return fail(QMV_ERR_CUDA, "cannot locate the device error word");

  const size_t smem = kSmemL;
  b.smem_bytes = (uint32_t)smem;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.blockDim = dim3(kThreadsL);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  int workers = 0;
  rc = workers_for(C, &workers);
  if (rc) return rc;
  workers = (int)std::min<int64_t>(std::min(workers, kMaxWorkersL), n_units);
  b.n_workers = workers;

  // largest units first, each to the least loaded worker
  if (n_units <= kMaxUnitsL && !same_cost) {
    std::vector<std::pair<int64_t, int>> cost((size_t)n_units);
    for (int i = 0; i < n; ++i) {
      const LutTask& T = b.t[i];
      const int nu = (T.N + T.rows - 1) / T.rows;
      for (int u = 0; u < nu; ++u) {
        const int64_t r = std::min(T.rows, T.N - u * T.rows);
        cost[(size_t)(T.unit0 + u)] = {r * T.KB, T.unit0 + u};
      }
    }
    std::stable_sort(cost.begin(), cost.end(), [](const auto& a, const auto& c) { return a.first > c.first; });
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int w = 0; w < workers; ++w) heap.push({0, w});
    std::vector<std::vector<int>> lists((size_t)workers);
    for (const auto& c : cost) {
      Load l = heap.top();
      heap.pop();
      lists[(size_t)l.second].push_back(c.second);
      l.first += c.first;
      heap.push(l);
    }
    int pos = 0;
    for (int w = 0; w < workers; ++w) {
      b.sched_off[w] = (uint16_t)pos;
      for (int u : lists[(size_t)w]) b.sched[pos++] = (uint16_t)u;
    }
    b.sched_off[workers] = (uint16_t)pos;
    b.sched_n = pos;
  } else {
    b.sched_n = 0;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = ++na;
  }
  cfg.gridDim = dim3((unsigned)(workers * C));
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, b);
  if (e != cudaSuccess) return cuda_fail(e, "lookup matvec launch");
  return QMV_OK;
}

}  // namespace

int run_lut(const qmv_task* tasks, int n, cudaStream_t s) {
  static thread_local LutBatch b;
  if (n < 1 || n > kMaxTasks) return fail(QMV_ERR_ARG, "n_tasks=%d outside 1..%d", n, kMaxTasks);
  if (!tasks || !tasks[0].desc) return fail(QMV_ERR_ARG, "NULL task or desc");
  const uint32_t fmt = tasks[0].desc->format;
  int min_kb = 1 << 30;
  for (int i = 0; i < n; ++i) {
    const qmv_task& t = tasks[i];
    int rc = check_lut_desc(t.desc);
    if (rc) return fail(rc, "task %d: %s", i, qmv_last_error());
    if (t.desc->format != fmt) return fail(QMV_ERR_ARG, "task %d: one launch serves one lookup layout", i);
    if (!t.w || !t.x || !t.y) return fail(QMV_ERR_ARG, "task %d: NULL w, x or y", i);
    if (!aligned16(t.w) || !aligned16(t.x) || !aligned16(t.y))
      return fail(QMV_ERR_ALIGN, "task %d: w, x and y must be 16-byte aligned", i);
    LutTask& T = b.t[i];
    T.codes = static_cast<const unsigned char*>(t.w) + t.desc->off[0];
    T.x = static_cast<const uint16_t*>(t.x);
    T.y = t.y;
    T.N = (int32_t)t.desc->N;
    T.rows = kUnitRowsMax;
    T.KB = (int32_t)(t.desc->K / QMV_GROUP);
    min_kb = std::min(min_kb, T.KB);
  }
  return fmt == QMV_INT4_LUT ? launch_lut<QMV_INT4_LUT, 0>(b, n, min_kb, s, false)
                              : launch_lut<QMV_TERNARY2_LUT, 0>(b, n, min_kb, s, false);
}

int run_lut_moe(const LutMoeCall& c, cudaStream_t s) {
  static thread_local LutBatch b;
  const int P = c.M * c.topk;
  LutMoe& mo = b.moe;
  mo.routing = MoeRouting{c.logits, c.E, c.topk, c.M};
  mo.x = c.x;
  mo.y = c.y;
  mo.gu = reinterpret_cast<float*>(c.ws + c.off_gu);
  mo.ws = c.ws;
  mo.off_slot_expert = c.off_slot_expert;
  mo.off_slot_first = c.off_slot_first;
  mo.off_slot_count = c.off_slot_count;
  mo.off_pair_token = c.off_pair_token;
  mo.off_pair_prob = c.off_pair_prob;
  mo.stride = c.stride;
  mo.I = (int32_t)c.I;
  mo.H = (int32_t)c.H;
  mo.ldx = (int32_t)c.ldx;
  mo.ldy = (int32_t)c.ldy;
  // gate|up: pair i reads its expert's [gate; up] matrix (2I x H) and writes g|u
  for (int i = 0; i < P; ++i) {
    LutTask& T = b.t[i];
    T.codes = c.gu_codes;
    T.x = nullptr;
    T.y = nullptr;
    T.N = (int32_t)(2 * c.I);
    T.rows = kUnitRowsMax;
    T.KB = (int32_t)(c.H / QMV_GROUP);
  }
  int rc = launch_lut<QMV_TERNARY2_LUT, 1>(b, P, (int)(c.H / QMV_GROUP), s, false);
  if (rc) return rc;
  // down: pair i reads its expert's down matrix (H x I) and adds p * W_down h into y
  for (int i = 0; i < P; ++i) {
    LutTask& T = b.t[i];
    T.codes = c.dn_codes;
    T.N = (int32_t)c.H;
    T.rows = kUnitRowsMax;
    T.KB = (int32_t)(c.I / QMV_GROUP);
  }
  return launch_lut<QMV_TERNARY2_LUT, 2>(b, P, (int)(c.I / QMV_GROUP), s, true);
}

}  // namespace qmv
