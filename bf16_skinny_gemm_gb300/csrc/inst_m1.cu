// Kernel instantiations for M = 1 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(1, kKernelsM1)
}  // namespace sk
