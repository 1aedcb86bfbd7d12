// k_tc.cu -- tensor-core (tcgen05) variants; placeholder until implemented.
#include "cbs_internal.cuh"

namespace cbs {
cbs_status plan_tc(cbs_plan_t &p) {
    return fail(CBS_ERR_UNSUPPORTED, "tensor-core variant %d not built yet", p.variant);
}
cbs_status launch_tc(const cbs_plan_t &p, const void *, const void *, const void *, const float *,
                     float, void *, void *, cudaStream_t) {
    return fail(CBS_ERR_UNSUPPORTED, "tensor-core variant %d not built yet", p.variant);
}
}  // namespace cbs
