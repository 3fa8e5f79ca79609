// Instantiation of the varlen forward kernel for d_qk = 96, d_v = 96.
#include "varlen_fwd_kernel.cuh"
FA_DEFINE_VARLEN_LAUNCHER(96, 96)
