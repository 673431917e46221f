// Kernel instantiations for M = 4 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(4, kKernelsM4)
}  // namespace sk
