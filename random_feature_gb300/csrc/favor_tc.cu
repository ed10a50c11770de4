// Tensor-core (tcgen05) path: placeholder until the sm_103a kernels land.
#include "favor_internal.h"

namespace favor {

bool tc_supported(const Handle&) { return false; }

favor_status tc_feature_map(const Handle&, const void*, void*, int, int, cudaStream_t) {
    return set_error(FAVOR_ERR_UNSUPPORTED, "tensor-core path not built");
}
favor_status tc_bidir(const Handle&, const void*, const void*, const void*, void*, int, int, cudaStream_t) {
    return set_error(FAVOR_ERR_UNSUPPORTED, "tensor-core path not built");
}
favor_status tc_causal(const Handle&, const void*, const void*, const void*, void*, int, int, cudaStream_t) {
    return set_error(FAVOR_ERR_UNSUPPORTED, "tensor-core path not built");
}

}  // namespace favor
