// Kernel instantiations for M = 2 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(2, kKernelsM2)
}  // namespace sk
