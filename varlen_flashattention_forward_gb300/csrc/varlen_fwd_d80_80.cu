// Instantiation of the varlen forward kernel for d_qk = 80, d_v = 80.
#include "varlen_fwd_kernel.cuh"
FA_DEFINE_VARLEN_LAUNCHER(80, 80)
