// argreduce kernels instantiated for one element type (f64).
#include "kernels_impl.cuh"

ARGR_DEFINE_LAUNCHERS(f64, argr::TagF64)
