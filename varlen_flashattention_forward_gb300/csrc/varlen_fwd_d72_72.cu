// Instantiation of the varlen forward kernel for d_qk = 72, d_v = 72.
#include "varlen_fwd_kernel.cuh"
FA_DEFINE_VARLEN_LAUNCHER(72, 72)
