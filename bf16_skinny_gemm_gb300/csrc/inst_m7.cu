// Kernel instantiations for M = 7 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(7, kKernelsM7)
}  // namespace sk
