// The compiled configurations of the weight-streaming kernel.  Each line is
// (M, rows per lane group R, lanes per row LPR, loads per batch U, FMA mode
// (0 widened, 1 mixed precision, 2 packed FP32x2, 3 tensor cores on the diagonal of
// mma.sync), double-buffered batches);
// every configuration exists for M = 1..8.  The host
// library enumerates these as plans (times two CTA sizes) and the offline
// sweep times all of them.
#pragma once

#include "skinny_ldg.cuh"
#include "skinny_mma.cuh"
#include "skinny_tc05.cuh"

#define SK_LDG_CONFIGS(X, M)   \
    X(M, 1, 32, 8, 0, false)   \
    X(M, 1, 32, 8, 1, false)   \
    X(M, 1, 32, 4, 1, false)   \
    X(M, 2, 32, 2, 1, false)   \
    X(M, 2, 32, 4, 1, false)   \
    X(M, 4, 32, 2, 1, false)   \
    X(M, 2, 16, 2, 1, false)   \
    X(M, 1, 16, 4, 1, false)   \
    X(M, 4, 8, 2, 1, false)    \
    X(M, 1, 32, 4, 1, true)    \
    X(M, 2, 32, 2, 1, true)    \
    X(M, 2, 16, 2, 1, true)    \
    X(M, 1, 32, 8, 2, false)   \
    X(M, 2, 32, 4, 2, false)   \
    X(M, 4, 32, 2, 2, false)   \
    X(M, 2, 32, 2, 2, false)   \
    X(M, 4, 32, 4, 2, false)   \
    X(M, 2, 16, 2, 2, false)   \
    X(M, 1, 16, 4, 2, false)   \
    X(M, 4, 8, 2, 2, false)    \
    X(M, 2, 32, 2, 2, true)    \
    X(M, 1, 32, 8, 3, false)   \
    X(M, 2, 32, 4, 3, false)   \
    X(M, 4, 32, 2, 3, false)   \
    X(M, 2, 32, 2, 3, false)   \
    X(M, 4, 32, 4, 3, false)   \
    X(M, 1, 32, 4, 3, true)    \
    X(M, 2, 32, 2, 3, true)

// The same kernel reading x straight from global memory (no staging): (M, R,
// LPR, U, FMA mode).
#define SK_LDGX_CONFIGS(X, M)  \
    X(M, 1, 32, 8, 1)          \
    X(M, 2, 32, 4, 1)          \
    X(M, 4, 32, 2, 1)          \
    X(M, 2, 32, 2, 1)          \
    X(M, 1, 32, 4, 1)          \
    X(M, 2, 16, 2, 1)          \
    X(M, 4, 32, 2, 2)          \
    X(M, 2, 32, 4, 2)

#define SK_LDGX_ENTRY(M, R, LPR, U, FMODE)                                                 \
    {(FMODE) == 2 ? SGEMM_VARIANT_LDGX_FFMA2 : SGEMM_VARIANT_LDGX_MIXFMA, M, R, LPR, U, 1, \
     reinterpret_cast<const void *>(&skinny_ldg_kernel<M, R, LPR, U, FMODE, false, true>)},

#define SK_LDG_ENTRY(M, R, LPR, U, FMODE, DB)                                              \
    {(FMODE) == 3   ? SGEMM_VARIANT_LDG_MMA                                               \
     : (FMODE) == 2 ? SGEMM_VARIANT_LDG_FFMA2                                             \
                    : ((FMODE) == 1 ? SGEMM_VARIANT_LDG_MIXFMA : SGEMM_VARIANT_LDG),      \
     M, R, LPR, U, (DB) ? 2 : 1,                                                          \
     reinterpret_cast<const void *>(&skinny_ldg_kernel<M, R, LPR, U, FMODE, DB>)},

// Cluster-split instantiations of mixed-precision configurations (M, R, LPR,
// U, double-buffered): the split CTAs of a row range form a thread-block
// cluster and rank 0 adds the partial sums (SGEMM_VARIANT_LDG_CLUSTER).
#define SK_LDGCL_CONFIGS(X, M) \
    X(M, 1, 32, 8, false)      \
    X(M, 1, 32, 4, true)       \
    X(M, 2, 32, 4, false)      \
    X(M, 2, 32, 2, true)       \
    X(M, 4, 32, 2, false)

#define SK_LDGCL_ENTRY(M, R, LPR, U, DB)                             \
    {SGEMM_VARIANT_LDG_CLUSTER, M, R, LPR, U, (DB) ? 2 : 1,          \
     reinterpret_cast<const void *>(&skinny_ldg_kernel<M, R, LPR, U, 1, DB, false, true>)},

// Tensor-core configurations: (M, k-blocks per batch U, double-buffered).
// R = 16 rows per tile, 4 lanes share a row segment.
#define SK_MMA_CONFIGS(X, M) \
    X(M, 2, false)           \
    X(M, 4, false)           \
    X(M, 8, false)           \
    X(M, 1, true)            \
    X(M, 2, true)            \
    X(M, 4, true)

#define SK_MMA_ENTRY(M, U, DB)                          \
    {SGEMM_VARIANT_MMA, M, 16, 4, U, (DB) ? 2 : 1,      \
     reinterpret_cast<const void *>(&skinny_mma_kernel<M, U, DB>)},

// TMA + tcgen05 kernel: one instantiation per M; tile rows 128, and the ring
// depth, boxes per stage and cluster split are launch parameters (U = 0,
// stages = 0 mark "any").
#define SK_TC05_ENTRY(M) \
    {SGEMM_VARIANT_TC05, M, 128, 0, 0, 0, reinterpret_cast<const void *>(&tc05::skinny_tc05_kernel<M>)},

#define SK_DEFINE_TABLE(M, NAME)                                                          \
    const KernelInfo NAME[] = {SK_LDG_CONFIGS(SK_LDG_ENTRY, M) SK_MMA_CONFIGS(SK_MMA_ENTRY, M) \
                                   SK_LDGX_CONFIGS(SK_LDGX_ENTRY, M)                       \
                                       SK_LDGCL_CONFIGS(SK_LDGCL_ENTRY, M) SK_TC05_ENTRY(M)};
