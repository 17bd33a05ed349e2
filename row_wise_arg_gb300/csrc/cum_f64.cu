// cummax / cummin with indices, instantiated for one element type (f64).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(f64, argr::CumF64)
