// Mixture-of-experts decode over ternary SwiGLU experts.
#include "qmv_internal.cuh"

using namespace qmv;

extern "C" {

size_t moe_workspace_size(int, int, int, int64_t, int64_t) { return 0; }

int moe_qmv_run(const qmv_desc*, const qmv_desc*, const void*, int64_t, int64_t, int, const float*, int,
                const void*, int, int64_t, float*, int64_t, void*, size_t, void*) {
  return fail(QMV_ERR_UNSUPPORTED, "moe_qmv_run: not built yet");
}

}  // extern "C"
