// Non-last-axis ArgMax/ArgMin kernels instantiated for one element type (f32).
#include "kernels_impl.cuh"

ARGR_DEFINE_AXIS_LAUNCHER(f32, argr::TagF32)
