// Kernel instantiations for M = 5 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(5, kKernelsM5)
}  // namespace sk
