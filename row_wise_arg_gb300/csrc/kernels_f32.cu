// argreduce kernels instantiated for one element type (f32).
#include "kernels_impl.cuh"

ARGR_DEFINE_LAUNCHERS(f32, argr::TagF32)
