// The compiled configurations of the weight-streaming kernel.  Each line is
// (M, rows per lane group R, lanes per row LPR, loads in flight per lane U,
// mixed-precision FMA); every configuration exists for M = 1..4.  The host
// library enumerates these as plans (times two CTA sizes) and the offline
// sweep times all of them.
#pragma once

#include "skinny_ldg.cuh"
#include "skinny_mma.cuh"

#define SK_LDG_CONFIGS(X, M)   \
    X(M, 1, 32, 8, false)      \
    X(M, 2, 32, 4, false)      \
    X(M, 1, 32, 8, true)       \
    X(M, 1, 32, 4, true)       \
    X(M, 1, 32, 16, true)      \
    X(M, 2, 32, 2, true)       \
    X(M, 2, 32, 4, true)       \
    X(M, 4, 32, 2, true)       \
    X(M, 2, 16, 2, true)       \
    X(M, 1, 16, 4, true)       \
    X(M, 4, 8, 2, true)

#define SK_LDG_ENTRY(M, R, LPR, U, MIX)                                                  \
    {(MIX) ? SGEMM_VARIANT_LDG_MIXFMA : SGEMM_VARIANT_LDG, M, R, LPR, U,                 \
     reinterpret_cast<const void *>(&skinny_ldg_kernel<M, R, LPR, U, MIX>)},

// Tensor-core configurations: (M, k-blocks per batch U).  R = 16 rows per tile,
// 4 lanes share a row segment.
#define SK_MMA_CONFIGS(X, M) \
    X(M, 2)                  \
    X(M, 4)                  \
    X(M, 8)

#define SK_MMA_ENTRY(M, U) \
    {SGEMM_VARIANT_MMA, M, 16, 4, U, reinterpret_cast<const void *>(&skinny_mma_kernel<M, U>)},

#define SK_DEFINE_TABLE(M, NAME) \
    const KernelInfo NAME[] = {SK_LDG_CONFIGS(SK_LDG_ENTRY, M) SK_MMA_CONFIGS(SK_MMA_ENTRY, M)};
