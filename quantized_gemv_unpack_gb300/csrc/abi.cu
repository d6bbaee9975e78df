// Host side of the C ABI: error reporting, layout descriptors, argument
// checks and dispatch of the matvec entry points.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "lut.cuh"

namespace qmv {

// Per-device status word written by kernels that meet corrupt packed data
// (first error wins). Read and cleared by qmv_check_status.
__device__ int g_qmv_error_word;

namespace {
thread_local char g_msg[512] = "";
std::mutex g_mu;
std::vector<int*> g_err_ptr;     // per device ordinal
std::vector<int> g_sms;          // per device ordinal

struct FitEntry {
  int dev;
  const void* kernel;
  int threads;
  size_t smem;
  int per_sm;
};
std::vector<FitEntry> g_fit;
// the largest dynamic shared memory size a kernel has been allowed on a device:
// the attribute is only ever raised, so a smaller launch cannot lower it under
// a larger cached one
struct SmemAttr {
  int dev;
  const void* kernel;
  size_t smem;
};
std::vector<SmemAttr> g_smem_attr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}
}  // namespace

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(QMV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int* device_error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_err_ptr.size() <= d) g_err_ptr.resize(d + 1, nullptr);
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qmv_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<int*>(p);
  }
  return g_err_ptr[d];
}

int sm_count() {
  const int d = current_device();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_sms.size() <= d) g_sms.resize(d + 1, 0);
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

int kernel_fit(const void* kernel, int threads, size_t smem, int* per_sm) {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  for (const FitEntry& f : g_fit)
    if (f.dev == d && f.kernel == kernel && f.threads == threads && f.smem == smem) {
      *per_sm = f.per_sm;
      return QMV_OK;
    }
  if (smem > 48 * 1024) {
    SmemAttr* a = nullptr;
    for (SmemAttr& x : g_smem_attr)
      if (x.dev == d && x.kernel == kernel) a = &x;
    if (!a || a->smem < smem) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
      if (a) a->smem = smem;
      else g_smem_attr.push_back({d, kernel, smem});
    }
  }
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (n < 1) return fail(QMV_ERR_UNSUPPORTED, "kernel with %d threads and %zu B shared memory does not fit an SM", threads, smem);
  g_fit.push_back({d, kernel, threads, smem, n});
  *per_sm = n;
  return QMV_OK;
}

namespace {

int64_t align256(int64_t n) { return (n + 255) / 256 * 256; }

void fill_sections(qmv_desc* d, const int64_t* sizes, int n) {
  int64_t pos = 0;
  for (int i = 0; i < QMV_MAX_SECTIONS; ++i) {
    d->off[i] = 0;
    d->bytes[i] = 0;
  }
  for (int i = 0; i < n; ++i) {
    d->off[i] = pos;
    d->bytes[i] = sizes[i];
    pos = align256(pos + sizes[i]);
  }
  d->total_bytes = pos;
}

}  // namespace

int check_desc(const qmv_desc* d, int format) {
  if (!d) return fail(QMV_ERR_ARG, "desc is NULL");
  if (d->abi_version != QMV_ABI_VERSION)
    return fail(QMV_ERR_ARG, "desc abi_version %u, library %d", d->abi_version, QMV_ABI_VERSION);
  if ((int)d->format != format) return fail(QMV_ERR_ARG, "desc format %u, call expects %d", d->format, format);
  if (d->N <= 0 || d->K <= 0) return fail(QMV_ERR_ARG, "desc N=%lld K=%lld", (long long)d->N, (long long)d->K);
  if (format == QMV_TERNARY2 || format == QMV_INT4) {
    if (d->group != QMV_GROUP || d->K % QMV_GROUP) return fail(QMV_ERR_ARG, "K=%lld must be a multiple of 128", (long long)d->K);
    if (d->N > INT32_MAX / 2 || d->K > (1 << 26)) return fail(QMV_ERR_UNSUPPORTED, "matrix too large");
    qmv_desc ref;
    qmv_pack_desc(format, d->N, d->K, d->group, &ref);
    for (int i = 0; i < 2; ++i)
      if (ref.off[i] != d->off[i] || ref.bytes[i] != d->bytes[i])
        return fail(QMV_ERR_ARG, "desc section %d does not match the layout of a %lld x %lld matrix", i,
                    (long long)d->N, (long long)d->K);
  }
  return QMV_OK;
}

int build_task(const qmv_desc* d, int format, const void* w, const void* x, int64_t ldx, float* y, int64_t ldy,
               GemvTask* t) {
  int rc = check_desc(d, format);
  if (rc) return rc;
  if (!w || !x || !y) return fail(QMV_ERR_ARG, "NULL w, x or y");
  if (!aligned16(w) || !aligned16(x) || !aligned16(y)) return fail(QMV_ERR_ALIGN, "w, x and y must be 16-byte aligned");
  if (ldx < d->K || ldy < d->N) return fail(QMV_ERR_ARG, "ldx=%lld < K or ldy=%lld < N", (long long)ldx, (long long)ldy);
  if (ldx % 8) return fail(QMV_ERR_ALIGN, "ldx=%lld must be a multiple of 8 (16-byte rows)", (long long)ldx);
  if (ldx > INT32_MAX || ldy > INT32_MAX) return fail(QMV_ERR_UNSUPPORTED, "leading dimension too large");
  const char* base = static_cast<const char*>(w);
  t->codes = reinterpret_cast<const uint32_t*>(base + d->off[0]);
  t->scales = reinterpret_cast<const uint16_t*>(base + d->off[1]);
  t->x = static_cast<const uint16_t*>(x);
  t->y = y;
  t->N = (int32_t)d->N;
  t->K = (int32_t)d->K;
  t->ldx = (int32_t)ldx;
  t->ldy = (int32_t)ldy;
  t->tile0 = 0;
  t->pad = 0;
  return QMV_OK;
}

namespace {

// Launch `n` tasks with M activation rows: one tensor-core launch, or
// fp16-FMA launches of <= 8 rows each. `flags` holds the QMV_FLAG_PATH_* bits
// of the tasks' descriptors.
int run_tasks(int format, GemvTask* tasks, int n, int M, uint64_t flags, cudaStream_t s) {
  static thread_local GemvBatch b;
  const uint64_t path = flags & (QMV_FLAG_PATH_FMA | QMV_FLAG_PATH_MMA);
  if (path == (QMV_FLAG_PATH_FMA | QMV_FLAG_PATH_MMA)) return fail(QMV_ERR_ARG, "both QMV_FLAG_PATH_FMA and _MMA set");
  if (flags & ~(uint64_t)(QMV_FLAG_PATH_FMA | QMV_FLAG_PATH_MMA | QMV_FLAG_TEST_WAIT_TIMEOUT))
    return fail(QMV_ERR_ARG, "unknown qmv_desc.flags bits 0x%llx", (unsigned long long)flags);
  b.test_wait_us = (flags & QMV_FLAG_TEST_WAIT_TIMEOUT) ? 1000u : 0u;
  if (path == QMV_FLAG_PATH_MMA || (path == 0 && M >= mma_min_m(format))) {
    for (int i = 0; i < n; ++i) b.t[i] = tasks[i];
    b.n_tasks = n;
    return launch_gemv_mma(format, b, M, s);
  }
  for (int m0 = 0; m0 < M; m0 += 8) {
    const int mt = M - m0 < 8 ? M - m0 : 8;
    for (int i = 0; i < n; ++i) {
      GemvTask t = tasks[i];
      t.x += (size_t)m0 * t.ldx;
      t.y += (size_t)m0 * t.ldy;
      b.t[i] = t;
    }
    b.n_tasks = n;
    int rc = launch_gemv(format, b, mt, s);
    if (rc) return rc;
  }
  return QMV_OK;
}

int run_one(int format, const qmv_desc* d, const void* w, const void* x, int M, int64_t ldx, float* y, int64_t ldy,
            void* stream) {
  if (M < 1 || M > QMV_MAX_M) return fail(QMV_ERR_ARG, "M=%d outside 1..%d", M, QMV_MAX_M);
  GemvTask t;
  int rc = build_task(d, format, w, x, ldx, y, ldy, &t);
  if (rc) return rc;
  return run_tasks(format, &t, 1, M, d->flags, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace qmv

using namespace qmv;

extern "C" {

const char* qmv_last_error(void) { return g_msg; }

int qmv_pack_desc(int format, int64_t N, int64_t K, int32_t group, qmv_desc* out) {
  if (!out) return fail(QMV_ERR_ARG, "out is NULL");
  if (format == QMV_CASS) return fail(QMV_ERR_UNSUPPORTED, "Cassandra layouts depend on the data; use cass_pack_host");
  if (format == QMV_CASS_MX) {
    // Cassandra-2 (MX): fixed layout, see qmv.h
    if (group != 32) return fail(QMV_ERR_ARG, "group must be 32 for QMV_CASS_MX");
    if (N <= 0 || K <= 0 || K % 64) return fail(QMV_ERR_ARG, "N=%lld K=%lld (K must be a positive multiple of 64)", (long long)N, (long long)K);
    memset(out, 0, sizeof(*out));
    out->abi_version = QMV_ABI_VERSION;
    out->format = (uint32_t)format;
    out->N = N;
    out->K = K;
    out->group = group;
    const int64_t sizes[6] = {N * K / 8, N * K / 64, N * K / 16, N * K / 4, N * K / 4, N * K};
    fill_sections(out, sizes, 6);
    return QMV_OK;
  }
  if (format == QMV_TERNARY2_LUT || format == QMV_INT4_LUT) {
    // byte-lookup layouts, see qmv.h: 1 KB (ternary) or 2 KB (INT4) records of
    // (block, 32-row group), scales [KB][NG * 32]
    if (group != QMV_GROUP) return fail(QMV_ERR_ARG, "group must be 128");
    if (N <= 0 || K <= 0 || K % QMV_GROUP) return fail(QMV_ERR_ARG, "N=%lld K=%lld (K must be a positive multiple of 128)", (long long)N, (long long)K);
    memset(out, 0, sizeof(*out));
    out->abi_version = QMV_ABI_VERSION;
    out->format = (uint32_t)format;
    out->N = N;
    out->K = K;
    out->group = group;
    const int64_t NG = (N + 31) / 32, KB = K / QMV_GROUP;
    const int64_t sizes[2] = {NG * KB * (format == QMV_INT4_LUT ? 2048 : 1024), KB * NG * 32 * 2};
    fill_sections(out, sizes, 2);
    return QMV_OK;
  }
  if (format != QMV_TERNARY2 && format != QMV_INT4) return fail(QMV_ERR_ARG, "unknown format %d", format);
  if (group != QMV_GROUP) return fail(QMV_ERR_ARG, "group must be 128");
  if (N <= 0 || K <= 0 || K % QMV_GROUP) return fail(QMV_ERR_ARG, "N=%lld K=%lld (K must be a positive multiple of 128)", (long long)N, (long long)K);
  memset(out, 0, sizeof(*out));
  out->abi_version = QMV_ABI_VERSION;
  out->format = (uint32_t)format;
  out->N = N;
  out->K = K;
  out->group = group;
  const int64_t padded = (N + 15) / 16 * 16;   // row groups of 16
  const int64_t codes = format == QMV_TERNARY2 ? padded * K / 4 : padded * K / 2;
  const int64_t sizes[2] = {codes, padded / 16 * scale_steps(K) * 256};
  fill_sections(out, sizes, 2);
  return QMV_OK;
}

int qmv_run_ternary(const qmv_desc* desc, const void* w, const void* x_bf16, int M, int64_t ldx, float* y,
                    int64_t ldy, void* stream) {
  if (desc && (desc->format == QMV_TERNARY2_SPARSE || desc->format == QMV_TERNARY2_LUT)) {
    qmv_task t{desc, w, x_bf16, y, ldx, ldy};
    return qmv_run_batch((int)desc->format, &t, 1, M, stream);
  }
  return run_one(QMV_TERNARY2, desc, w, x_bf16, M, ldx, y, ldy, stream);
}

int qmv_run_int4(const qmv_desc* desc, const void* w, const void* x_bf16, int M, int64_t ldx, float* y,
                 int64_t ldy, void* stream) {
  if (desc && desc->format == QMV_INT4_LUT) {
    qmv_task t{desc, w, x_bf16, y, ldx, ldy};
    return qmv_run_batch(QMV_INT4_LUT, &t, 1, M, stream);
  }
  return run_one(QMV_INT4, desc, w, x_bf16, M, ldx, y, ldy, stream);
}

int qmv_run_batch(int format, const qmv_task* tasks, int n_tasks, int M, void* stream) {
  if (format == QMV_TERNARY2_LUT || format == QMV_INT4_LUT) {
    if (!tasks || n_tasks < 1 || n_tasks > QMV_MAX_BATCH) return fail(QMV_ERR_ARG, "n_tasks=%d outside 1..%d", n_tasks, QMV_MAX_BATCH);
    if (M != 1) return fail(QMV_ERR_UNSUPPORTED, "the lookup layout serves M = 1 (got M=%d)", M);
    for (int i = 0; i < n_tasks; ++i)
      if (!tasks[i].desc || (int)tasks[i].desc->format != format)
        return fail(QMV_ERR_ARG, "task %d: descriptor format differs from the batch's", i);
    return run_lut(tasks, n_tasks, static_cast<cudaStream_t>(stream));
  }
  if (format == QMV_TERNARY2_SPARSE) {
    if (!tasks || n_tasks < 1 || n_tasks > QMV_MAX_BATCH) return fail(QMV_ERR_ARG, "n_tasks=%d outside 1..%d", n_tasks, QMV_MAX_BATCH);
    if (M < 1 || M > 8) return fail(QMV_ERR_ARG, "sparse ternary: M=%d outside 1..8", M);
    static thread_local const qmv_desc* ds[QMV_MAX_BATCH];
    static thread_local const void* ws[QMV_MAX_BATCH];
    static thread_local const void* xs[QMV_MAX_BATCH];
    static thread_local float* ys[QMV_MAX_BATCH];
    static thread_local int64_t lx[QMV_MAX_BATCH], ly[QMV_MAX_BATCH];
    for (int i = 0; i < n_tasks; ++i) {
      const qmv_task& t = tasks[i];
      int rc = check_sparse_desc(t.desc);
      if (rc) return fail(rc, "task %d: %s", i, qmv_last_error());
      if (!t.w || !t.x || !t.y) return fail(QMV_ERR_ARG, "task %d: NULL w, x or y", i);
      if (!aligned16(t.w) || !aligned16(t.x) || !aligned16(t.y)) return fail(QMV_ERR_ALIGN, "task %d: w, x and y must be 16-byte aligned", i);
      if (t.ldx < t.desc->K || t.ldy < t.desc->N || t.ldx % 8 || t.ldx > INT32_MAX || t.ldy > INT32_MAX)
        return fail(QMV_ERR_ARG, "task %d: ldx=%lld ldy=%lld", i, (long long)t.ldx, (long long)t.ldy);
      ds[i] = t.desc;
      ws[i] = t.w;
      xs[i] = t.x;
      ys[i] = t.y;
      lx[i] = t.ldx;
      ly[i] = t.ldy;
    }
    return run_sparse(ds, ws, xs, lx, ys, ly, n_tasks, M, static_cast<cudaStream_t>(stream));
  }
  if (format != QMV_TERNARY2 && format != QMV_INT4) return fail(QMV_ERR_UNSUPPORTED, "qmv_run_batch serves ternary and INT4");
  if (!tasks || n_tasks < 1 || n_tasks > QMV_MAX_BATCH) return fail(QMV_ERR_ARG, "n_tasks=%d outside 1..%d", n_tasks, QMV_MAX_BATCH);
  if (M < 1 || M > QMV_MAX_M) return fail(QMV_ERR_ARG, "M=%d outside 1..%d", M, QMV_MAX_M);
  static thread_local GemvTask t[QMV_MAX_BATCH];
  int64_t tiles = 0;
  uint64_t flags = 0;
  for (int i = 0; i < n_tasks; ++i) {
    int rc = build_task(tasks[i].desc, format, tasks[i].w, tasks[i].x, tasks[i].ldx, tasks[i].y, tasks[i].ldy, &t[i]);
    if (rc) return fail(rc, "task %d: %s", i, qmv_last_error());
    tiles += (t[i].N + 3) / 4;
    flags |= tasks[i].desc->flags;
  }
  if (tiles > INT32_MAX / 2) return fail(QMV_ERR_UNSUPPORTED, "batch too large");
  return run_tasks(format, t, n_tasks, M, flags, static_cast<cudaStream_t>(stream));
}

int qmv_check_status(void* stream, int32_t* device_code) {
  if (device_code) *device_code = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* p = device_error_word();
  if (!p) return fail(QMV_ERR_CUDA, "cannot locate the device error word");
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (v) {
    const int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  }
  if (device_code) *device_code = v;
  if (v) return fail(v, "a kernel reported status %d (%s)", v,
                     v == QMV_ERR_TIMEOUT ? "a bounded device wait gave up" : "corrupt packed data");
  return QMV_OK;
}

}  // extern "C"
