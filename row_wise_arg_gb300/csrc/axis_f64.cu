// Non-last-axis ArgMax/ArgMin kernels instantiated for one element type (f64).
#include "kernels_impl.cuh"

ARGR_DEFINE_AXIS_LAUNCHER(f64, argr::TagF64)
