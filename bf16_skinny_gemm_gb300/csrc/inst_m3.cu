// Kernel instantiations for M = 3 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(3, kKernelsM3)
}  // namespace sk
