// cummax / cummin with indices, instantiated for one element type (i32).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(i32, argr::CumI32)
