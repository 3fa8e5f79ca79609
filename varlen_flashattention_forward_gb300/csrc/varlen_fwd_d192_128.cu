// Instantiation of the varlen forward kernel for d_qk = 192, d_v = 128.
#include "varlen_fwd_kernel.cuh"
FA_DEFINE_VARLEN_LAUNCHER(192, 128)
