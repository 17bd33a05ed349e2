// Non-last-axis ArgMax/ArgMin kernels instantiated for one element type (f16).
#include "kernels_impl.cuh"

ARGR_DEFINE_AXIS_LAUNCHER(f16, argr::TagF16)
