// Split-K second-pass kernels (one per M) and the per-M kernel count.
#include "kernel_table.cuh"

namespace sk {

#define SK_COUNT_ONE(M, R, LPR, U, FMODE, DB) +1
#define SK_COUNT_MMA(M, U, DB) +1
#define SK_COUNT_LDGX(M, R, LPR, U, FMODE) +1
#define SK_COUNT_LDGCL(M, R, LPR, U, DB) +1
const int kKernelCountPerM = 0 SK_LDG_CONFIGS(SK_COUNT_ONE, 1) SK_MMA_CONFIGS(SK_COUNT_MMA, 1)
    SK_LDGX_CONFIGS(SK_COUNT_LDGX, 1) SK_LDGCL_CONFIGS(SK_COUNT_LDGCL, 1) + 1 /* TMA + tcgen05 */;

const void *const kReduceKernels[kMaxM + 1] = {
    nullptr,
    reinterpret_cast<const void *>(&splitk_reduce_kernel<1>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<2>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<3>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<4>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<5>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<6>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<7>),
    reinterpret_cast<const void *>(&splitk_reduce_kernel<8>),
};

}  // namespace sk
