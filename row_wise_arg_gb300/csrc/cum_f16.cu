// cummax / cummin with indices, instantiated for one element type (f16).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(f16, argr::CumF16)
