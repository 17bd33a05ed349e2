// cummax / cummin with indices, instantiated for one element type (i64).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(i64, argr::CumI64)
