// Kernel instantiations for M = 6 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(6, kKernelsM6)
}  // namespace sk
