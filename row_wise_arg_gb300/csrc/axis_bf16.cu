// Non-last-axis ArgMax/ArgMin kernels instantiated for one element type (bf16).
#include "kernels_impl.cuh"

ARGR_DEFINE_AXIS_LAUNCHER(bf16, argr::TagBF16)
