// Dispatch to the tcgen05 tensor-core kernels.
#include "nm_internal.h"

bool nm_tc_linear_supports(const nm_config& c);
cudaError_t nm_tc_linear_launch(const nm_config& c, const nm_args& a, cudaStream_t s);
bool nm_tc_mlp_supports(const nm_config& c);
cudaError_t nm_tc_mlp_launch(const nm_config& c, const nm_args& a, cudaStream_t s);
bool nm_tc_mlp_wide_supports(const nm_config& c);
bool nm_tc_linear64_supports(const nm_config& c);
cudaError_t nm_tc_linear64_launch(const nm_config& c, const nm_args& a, cudaStream_t s);
cudaError_t nm_tc_mlp_wide_launch(const nm_config& c, const nm_args& a, cudaStream_t s);
bool nm_tc_deep_supports(const nm_config& c);
size_t nm_tc_deep_scratch_bytes(const nm_config& c, int B, int H);
cudaError_t nm_tc_deep_launch(const nm_config& c, const nm_args& a, cudaStream_t s);

bool nm_tc_supports(const nm_config& c) {
    if (nm_layers(c) > 2) return nm_tc_deep_supports(c);
    return nm_tc_linear_supports(c) || nm_tc_linear64_supports(c) || nm_tc_mlp_supports(c) ||
           nm_tc_mlp_wide_supports(c);
}

// Kernels that can also write the per-token surprise (gradient norm).
bool nm_tc_supports_surprise(const nm_config& c) {
    if (nm_layers(c) > 2) return nm_tc_deep_supports(c);
    return nm_tc_linear_supports(c) || nm_tc_linear64_supports(c) || nm_tc_mlp_supports(c) ||
           nm_tc_mlp_wide_supports(c);
}

// Kernels that can record every chunk's start state (nm_args.ckpt) for the
// backward pass, without writing y.
bool nm_tc_supports_ckpt(const nm_config& c) { return nm_layers(c) <= 2 && nm_tc_linear_supports(c); }

// Only the deep-memory kernel keeps a per-unit workspace (the chunk's activations).
size_t nm_tc_scratch_bytes(const nm_config& c, int B, int H) {
    return nm_layers(c) > 2 && nm_tc_deep_supports(c) ? nm_tc_deep_scratch_bytes(c, B, H) : 0;
}

cudaError_t nm_tc_launch(const nm_config& c, const nm_args& a, cudaStream_t s, int num_sms, long long* launches) {
    (void)num_sms;
    cudaError_t e = cudaErrorNotSupported;
    if (nm_layers(c) > 2) e = nm_tc_deep_supports(c) ? nm_tc_deep_launch(c, a, s) : cudaErrorNotSupported;
    else if (nm_tc_linear_supports(c)) e = nm_tc_linear_launch(c, a, s);
    else if (nm_tc_linear64_supports(c)) e = nm_tc_linear64_launch(c, a, s);
    else if (nm_tc_mlp_supports(c)) e = nm_tc_mlp_launch(c, a, s);
    else if (nm_tc_mlp_wide_supports(c)) e = nm_tc_mlp_wide_launch(c, a, s);
    if (e == cudaSuccess) *launches += 1;
    return e;
}
