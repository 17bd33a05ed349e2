// argreduce kernels instantiated for one element type (bf16).
#include "kernels_impl.cuh"

ARGR_DEFINE_LAUNCHERS(bf16, argr::TagBF16)
