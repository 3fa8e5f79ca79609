// Instantiation of the varlen forward kernel for d_qk = 64, d_v = 64.
#include "varlen_fwd_kernel.cuh"
FA_DEFINE_VARLEN_LAUNCHER(64, 64)
