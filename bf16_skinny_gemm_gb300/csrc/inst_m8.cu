// Kernel instantiations for M = 8 (one translation unit per M so that the
// library builds in parallel).
#include "kernel_table.cuh"

namespace sk {
SK_DEFINE_TABLE(8, kKernelsM8)
}  // namespace sk
