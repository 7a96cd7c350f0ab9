// tcgen05 tensor-core kernels: dispatch.  (Kernels land in later files.)
#include "nm_internal.h"

bool nm_tc_supports(const nm_config& c) {
    (void)c;
    return false;
}

size_t nm_tc_scratch_bytes(const nm_config& c, int B, int H) {
    (void)c; (void)B; (void)H;
    return 0;
}

cudaError_t nm_tc_launch(const nm_config& c, const nm_args& a, cudaStream_t s, int num_sms, long long* launches) {
    (void)c; (void)a; (void)s; (void)num_sms; (void)launches;
    return cudaErrorNotSupported;
}
