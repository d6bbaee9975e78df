// Cassandra lossless bf16 split: host packer and GPU draft/target kernels.
#include "qmv_internal.cuh"

using namespace qmv;

extern "C" {

int cass_pack_host(const uint16_t*, int64_t, int64_t, const uint16_t*, int64_t, qmv_desc*, void*, int64_t) {
  return fail(QMV_ERR_UNSUPPORTED, "cass_pack_host: not built yet");
}

int cass_decode_draft(const qmv_desc*, const void*, const void*, int, int64_t, float*, int64_t, uint16_t*, void*) {
  return fail(QMV_ERR_UNSUPPORTED, "cass_decode_draft: not built yet");
}

int cass_reconstruct(const qmv_desc*, const void*, const void*, int, int64_t, float*, int64_t, uint16_t*, void*) {
  return fail(QMV_ERR_UNSUPPORTED, "cass_reconstruct: not built yet");
}

}  // extern "C"
