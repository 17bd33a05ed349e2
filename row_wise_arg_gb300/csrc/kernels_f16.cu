// argreduce kernels instantiated for one element type (f16).
#include "kernels_impl.cuh"

ARGR_DEFINE_LAUNCHERS(f16, argr::TagF16)
