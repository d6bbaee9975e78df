// Packed-weight files: a model's packed matrices in one file, written once
// after the offline packing step and loaded into caller-owned device memory
// ("Ternary Bonsai 2", section 3.6: the packed ternary indices, block scales
// and flags are exported as the model file that inference reads).
//
// File layout (little-endian; this library's format, version 1):
//   header   64 bytes at offset 0:
//              0  char[4]  magic "QMVF"
//              4  u32      version (1)
//              8  u32      n_tensors
//             12  u32      entry_bytes (sizeof(qmv_file_entry) = 288)
//             16  u64      table_offset (64)
//             24  u64      data_offset (first tensor, 4096-aligned)
//             32  u64      file_bytes
//             40  u32      table_crc   CRC-32 of the entry table
//             44  u32      header_crc  CRC-32 of bytes 0..43
//             48  16 bytes zero
//   table    n_tensors entries of entry_bytes at table_offset:
//              char[64] name (NUL-terminated), qmv_desc (flags 0), u64 offset
//              (4096-aligned), u64 bytes (= desc.total_bytes), u32 crc[8]
//              (CRC-32 of each section's desc.bytes[i] bytes, 0 for an absent
//              section)
//   data     each tensor's packed buffer at its offset, zero padding between.
// CRC-32 is the reflected polynomial 0xEDB88320 with initial value and final
// XOR 0xFFFFFFFF (the checksum of zip, PNG and Ethernet), computed here with
// eight 256-entry tables generated from the polynomial at first use.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "qmv_internal.cuh"

namespace qmv {
namespace {

constexpr char kMagic[4] = {'Q', 'M', 'V', 'F'};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kHeaderBytes = 64;
constexpr uint64_t kAlign = 4096;

struct Entry {
  char name[QMV_FILE_NAME_BYTES];
  qmv_desc desc;
  uint64_t offset;
  uint64_t bytes;
  uint32_t crc[QMV_MAX_SECTIONS];
};
static_assert(sizeof(qmv_desc) == 176, "qmv_desc is stored in files byte for byte");
static_assert(sizeof(Entry) == 288, "file entry size is part of the format");

uint32_t g_crc[8][256];
std::once_flag g_crc_once;

void crc_tables() {
  for (uint32_t i = 0; i < 256; ++i) {
    uint32_t c = i;
    for (int k = 0; k < 8; ++k) c = (c & 1u) ? (c >> 1) ^ 0xEDB88320u : c >> 1;
    g_crc[0][i] = c;
  }
  // table t advances a byte that is followed by t more bytes
  for (uint32_t i = 0; i < 256; ++i)
    for (int t = 1; t < 8; ++t) g_crc[t][i] = (g_crc[t - 1][i] >> 8) ^ g_crc[0][g_crc[t - 1][i] & 0xFFu];
}

uint32_t crc_update(uint32_t crc, const unsigned char* p, size_t n) {
  std::call_once(g_crc_once, crc_tables);
  uint32_t c = ~crc;
  while (n && (reinterpret_cast<uintptr_t>(p) & 7u)) {
    c = (c >> 8) ^ g_crc[0][(c ^ *p++) & 0xFFu];
    --n;
  }
  while (n >= 8) {
    uint32_t lo, hi;
    memcpy(&lo, p, 4);
    memcpy(&hi, p + 4, 4);
    lo ^= c;
    c = g_crc[7][lo & 0xFFu] ^ g_crc[6][(lo >> 8) & 0xFFu] ^ g_crc[5][(lo >> 16) & 0xFFu] ^ g_crc[4][lo >> 24] ^
        g_crc[3][hi & 0xFFu] ^ g_crc[2][(hi >> 8) & 0xFFu] ^ g_crc[1][(hi >> 16) & 0xFFu] ^ g_crc[0][hi >> 24];
    p += 8;
    n -= 8;
  }
  while (n--) c = (c >> 8) ^ g_crc[0][(c ^ *p++) & 0xFFu];
  return ~c;
}

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

void put_u32(unsigned char* p, uint32_t v) { memcpy(p, &v, 4); }
void put_u64(unsigned char* p, uint64_t v) { memcpy(p, &v, 8); }
uint32_t get_u32(const unsigned char* p) {
  uint32_t v;
  memcpy(&v, p, 4);
  return v;
}
uint64_t get_u64(const unsigned char* p) {
  uint64_t v;
  memcpy(&v, p, 8);
  return v;
}

// A descriptor as stored in a file: a known format whose sections lie inside
// its total size.
bool desc_is_sane(const qmv_desc& d) {
  if (d.abi_version != QMV_ABI_VERSION) return false;
  if (d.format < QMV_TERNARY2 || d.format > QMV_INT4_LUT) return false;
  if (d.N <= 0 || d.K <= 0 || d.total_bytes <= 0) return false;
  for (int i = 0; i < QMV_MAX_SECTIONS; ++i) {
    if (d.off[i] < 0 || d.bytes[i] < 0) return false;
    if (d.bytes[i] && d.off[i] + d.bytes[i] > d.total_bytes) return false;
  }
  return true;
}

bool write_all(int fd, const void* p, size_t n) {
  const char* c = static_cast<const char*>(p);
  while (n) {
    const ssize_t w = ::write(fd, c, n);
    if (w <= 0) return false;
    c += w;
    n -= (size_t)w;
  }
  return true;
}

}  // namespace
}  // namespace qmv

struct qmv_file {
  int fd;
  const unsigned char* map;
  uint64_t bytes;
  uint32_t n;
  const unsigned char* table;
};

using namespace qmv;

extern "C" {

uint32_t qmv_crc32(const void* data, size_t n, uint32_t crc) {
  if (!data) return crc;
  return crc_update(crc, static_cast<const unsigned char*>(data), n);
}

int qmv_file_write(const char* path, int n, const char* const* names, const qmv_desc* descs,
                   const void* const* buffers) {
  if (!path || n < 1 || !names || !descs || !buffers) return fail(QMV_ERR_ARG, "qmv_file_write: NULL argument or n < 1");
  std::vector<Entry> ents((size_t)n);
  uint64_t pos = align_up(kHeaderBytes + (uint64_t)n * sizeof(Entry), kAlign);
  const uint64_t data0 = pos;
  for (int i = 0; i < n; ++i) {
    Entry& e = ents[(size_t)i];
    memset(&e, 0, sizeof(e));
    if (!names[i] || strlen(names[i]) >= QMV_FILE_NAME_BYTES)
      return fail(QMV_ERR_ARG, "tensor %d: name missing or longer than %d bytes", i, QMV_FILE_NAME_BYTES - 1);
    for (int j = 0; j < i; ++j)
      if (strcmp(names[j], names[i]) == 0) return fail(QMV_ERR_ARG, "tensor name '%s' appears twice", names[i]);
    if (!buffers[i]) return fail(QMV_ERR_ARG, "tensor %d: NULL buffer", i);
    qmv_desc d = descs[i];
    d.flags = 0;
    if (!desc_is_sane(d)) return fail(QMV_ERR_ARG, "tensor '%s': descriptor is not a valid packed layout", names[i]);
    strncpy(e.name, names[i], QMV_FILE_NAME_BYTES - 1);
    e.desc = d;
    e.offset = pos;
    e.bytes = (uint64_t)d.total_bytes;
    const unsigned char* b = static_cast<const unsigned char*>(buffers[i]);
    for (int s = 0; s < QMV_MAX_SECTIONS; ++s)
      e.crc[s] = d.bytes[s] ? crc_update(0u, b + d.off[s], (size_t)d.bytes[s]) : 0u;
    pos = align_up(pos + e.bytes, kAlign);
  }
  unsigned char hdr[kHeaderBytes];
  memset(hdr, 0, sizeof(hdr));
  memcpy(hdr, kMagic, 4);
  put_u32(hdr + 4, kVersion);
  put_u32(hdr + 8, (uint32_t)n);
  put_u32(hdr + 12, (uint32_t)sizeof(Entry));
  put_u64(hdr + 16, kHeaderBytes);
  put_u64(hdr + 24, data0);
  put_u64(hdr + 32, pos);
  put_u32(hdr + 40, crc_update(0u, reinterpret_cast<const unsigned char*>(ents.data()), ents.size() * sizeof(Entry)));
  put_u32(hdr + 44, crc_update(0u, hdr, 44));

  const int fd = ::open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
  if (fd < 0) return fail(QMV_ERR_ARG, "cannot create %s", path);
  bool ok = write_all(fd, hdr, sizeof(hdr)) && write_all(fd, ents.data(), ents.size() * sizeof(Entry));
  uint64_t at = kHeaderBytes + ents.size() * sizeof(Entry);
  static const unsigned char zeros[kAlign] = {0};
  for (int i = 0; ok && i < n; ++i) {
    const Entry& e = ents[(size_t)i];
    ok = write_all(fd, zeros, (size_t)(e.offset - at)) && write_all(fd, buffers[i], (size_t)e.bytes);
    at = e.offset + e.bytes;
  }
  ok = ok && write_all(fd, zeros, (size_t)(pos - at));
  ok = (::close(fd) == 0) && ok;
  if (!ok) return fail(QMV_ERR_ARG, "writing %s failed", path);
  return QMV_OK;
}

int qmv_file_open(const char* path, qmv_file** out) {
  if (!path || !out) return fail(QMV_ERR_ARG, "qmv_file_open: NULL argument");
  *out = nullptr;
  const int fd = ::open(path, O_RDONLY);
  if (fd < 0) return fail(QMV_ERR_ARG, "cannot open %s", path);
  struct stat st;
  if (fstat(fd, &st) != 0 || st.st_size < (off_t)kHeaderBytes) {
    ::close(fd);
    return fail(QMV_ERR_CORRUPT, "%s: shorter than a qmv file header", path);
  }
  const uint64_t size = (uint64_t)st.st_size;
  void* m = mmap(nullptr, (size_t)size, PROT_READ, MAP_PRIVATE, fd, 0);
  if (m == MAP_FAILED) {
    ::close(fd);
    return fail(QMV_ERR_ARG, "%s: mmap failed", path);
  }
  const unsigned char* p = static_cast<const unsigned char*>(m);
  auto reject = [&](int status, const char* why) {
    munmap(m, (size_t)size);
    ::close(fd);
    return fail(status, "%s: %s", path, why);
  };
  if (memcmp(p, kMagic, 4) != 0) return reject(QMV_ERR_CORRUPT, "not a qmv file (magic)");
  if (get_u32(p + 44) != crc_update(0u, p, 44)) return reject(QMV_ERR_CORRUPT, "header CRC mismatch");
  if (get_u32(p + 4) != kVersion) return reject(QMV_ERR_UNSUPPORTED, "file version not supported by this library");
  const uint32_t n = get_u32(p + 8);
  const uint64_t tab = get_u64(p + 16);
  if (get_u32(p + 12) != sizeof(Entry) || tab != kHeaderBytes || n == 0 || n > (1u << 20))
    return reject(QMV_ERR_CORRUPT, "entry table description");
  if (get_u64(p + 32) != size) return reject(QMV_ERR_CORRUPT, "file size differs from the header's (truncated?)");
  if (tab + (uint64_t)n * sizeof(Entry) > size) return reject(QMV_ERR_CORRUPT, "entry table past the end");
  if (get_u32(p + 40) != crc_update(0u, p + tab, (size_t)n * sizeof(Entry)))
    return reject(QMV_ERR_CORRUPT, "entry table CRC mismatch");
  for (uint32_t i = 0; i < n; ++i) {
    Entry e;
    memcpy(&e, p + tab + (uint64_t)i * sizeof(Entry), sizeof(e));
    if (e.name[QMV_FILE_NAME_BYTES - 1] != 0 || !desc_is_sane(e.desc) || e.bytes != (uint64_t)e.desc.total_bytes ||
        e.offset % kAlign || e.offset < get_u64(p + 24) || e.offset + e.bytes > size)
      return reject(QMV_ERR_CORRUPT, "entry out of bounds or with an invalid descriptor");
  }
  qmv_file* f = static_cast<qmv_file*>(malloc(sizeof(qmv_file)));
  if (!f) return reject(QMV_ERR_ARG, "out of host memory");
  f->fd = fd;
  f->map = p;
  f->bytes = size;
  f->n = n;
  f->table = p + tab;
  *out = f;
  return QMV_OK;
}

int qmv_file_count(const qmv_file* f) { return f ? (int)f->n : 0; }

int qmv_file_tensor(const qmv_file* f, int index, char* name, qmv_desc* desc) {
  if (!f || index < 0 || (uint32_t)index >= f->n) return fail(QMV_ERR_ARG, "tensor index %d out of range", index);
  Entry e;
  memcpy(&e, f->table + (size_t)index * sizeof(Entry), sizeof(e));
  if (name) memcpy(name, e.name, QMV_FILE_NAME_BYTES);
  if (desc) *desc = e.desc;
  return QMV_OK;
}

int qmv_file_find(const qmv_file* f, const char* name) {
  if (!f || !name) return fail(QMV_ERR_ARG, "qmv_file_find: NULL argument");
  for (uint32_t i = 0; i < f->n; ++i)
    if (strncmp(reinterpret_cast<const char*>(f->table + (size_t)i * sizeof(Entry)), name, QMV_FILE_NAME_BYTES) == 0)
      return (int)i;
  return fail(QMV_ERR_ARG, "no tensor named '%s'", name);
}

// CRC check of every section of tensor `index`; the tensor's bytes on success.
static int checked_tensor(const qmv_file* f, int index, int64_t capacity, const unsigned char** src, uint64_t* bytes) {
  if (!f || index < 0 || (uint32_t)index >= f->n) return fail(QMV_ERR_ARG, "tensor index %d out of range", index);
  Entry e;
  memcpy(&e, f->table + (size_t)index * sizeof(Entry), sizeof(e));
  if (capacity < 0 || (uint64_t)capacity < e.bytes)
    return fail(QMV_ERR_ARG, "tensor '%s' needs %llu bytes, capacity %lld", e.name, (unsigned long long)e.bytes,
                (long long)capacity);
  const unsigned char* b = f->map + e.offset;
  for (int s = 0; s < QMV_MAX_SECTIONS; ++s)
    if (e.desc.bytes[s] && crc_update(0u, b + e.desc.off[s], (size_t)e.desc.bytes[s]) != e.crc[s])
      return fail(QMV_ERR_CORRUPT, "tensor '%s' section %d: CRC mismatch", e.name, s);
  *src = b;
  *bytes = e.bytes;
  return QMV_OK;
}

int qmv_file_read_host(const qmv_file* f, int index, void* dst, int64_t capacity) {
  if (!dst) return fail(QMV_ERR_ARG, "dst is NULL");
  const unsigned char* src = nullptr;
  uint64_t n = 0;
  int rc = checked_tensor(f, index, capacity, &src, &n);
  if (rc) return rc;
  memcpy(dst, src, (size_t)n);
  return QMV_OK;
}

int qmv_file_load(const qmv_file* f, int index, void* dst, int64_t capacity, void* stream) {
  if (!dst) return fail(QMV_ERR_ARG, "dst is NULL");
  if (!aligned16(dst)) return fail(QMV_ERR_ALIGN, "dst must be 16-byte aligned");
  const unsigned char* src = nullptr;
  uint64_t n = 0;
  int rc = checked_tensor(f, index, capacity, &src, &n);
  if (rc) return rc;
  // from pageable memory the call returns once the bytes are staged, so the
  // mapping may be closed afterwards
  cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)n, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy of a file tensor to the device");
  return QMV_OK;
}

void qmv_file_close(qmv_file* f) {
  if (!f) return;
  munmap(const_cast<unsigned char*>(f->map), (size_t)f->bytes);
  ::close(f->fd);
  free(f);
}

}  // extern "C"
