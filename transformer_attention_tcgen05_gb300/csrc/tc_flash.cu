// tcgen05 flash attention (bf16) -- under construction.
#include "common.cuh"
#include "kernels.h"

namespace attn {

bool tc_full_supported(int, int, int, int, int) { return false; }

attn_status_t tc_full(const Ctx &, const void *, const void *, const void *, void *, int, int,
                      int, int, int, float) {
    return ATTN_ERR_UNSUPPORTED;
}

bool tc_na3d_supported(int, int, int, int, int, int, const int *) { return false; }

attn_status_t tc_na3d(const Ctx &, const void *, const void *, const void *, void *, int, int,
                      int, int, int, int, const int *, float) {
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
