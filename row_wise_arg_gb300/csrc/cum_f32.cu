// cummax / cummin with indices, instantiated for one element type (f32).
#include "kernels_impl.cuh"
#include "cum_impl.cuh"

ARGR_DEFINE_CUM_LAUNCHER(f32, argr::CumF32)
