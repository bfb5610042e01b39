// attn_bwd_tc.cu -- bf16 striped causal attention backward on tcgen05.
#include "common.cuh"
#include "internal.h"

namespace striped {

int launch_tc_bwd(const void *, const void *, const void *, const void *, const float *, const void *, void *,
                  void *, void *, float *, float *, const AttnGeom &, int64_t *, cudaStream_t) {
    return STRIPED_ERR_UNSUPPORTED;
}

}  // namespace striped
