// cummax / cummin with indices, instantiated for one element type (bf16).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(bf16, argr::CumBF16)
