// The compiled configurations of the weight-streaming kernel.  Each line is
// (M, rows per lane group R, lanes per row LPR, loads in flight per row U);
// every configuration exists for M = 1..4.  The host library enumerates these
// as plans (times two CTA sizes) and the offline sweep times all of them.
#pragma once

#include "skinny_ldg.cuh"

#define SK_LDG_CONFIGS(X, M) \
    X(M, 1, 32, 4)           \
    X(M, 1, 32, 8)           \
    X(M, 2, 32, 2)           \
    X(M, 2, 32, 4)           \
    X(M, 4, 32, 2)           \
    X(M, 2, 16, 1)           \
    X(M, 1, 16, 2)           \
    X(M, 4, 8, 1)

#define SK_LDG_ENTRY(M, R, LPR, U) \
    {SGEMM_VARIANT_LDG, M, R, LPR, U, reinterpret_cast<const void *>(&skinny_ldg_kernel<M, R, LPR, U>)},

#define SK_DEFINE_TABLE(M, NAME) \
    const KernelInfo NAME[] = {SK_LDG_CONFIGS(SK_LDG_ENTRY, M)};
