// Geometry of the TMA + tcgen05 skinny-GEMM kernel (skinny_tc05.cuh), shared
// by the kernel and the host code that checks and launches its plans.
#pragma once

namespace sk {
namespace tc05 {

constexpr int kRows = 128;                      // rows of W per tile (MMA M)
constexpr int kCols = 16;                       // MMA N: rows of x, zero-padded
constexpr int kBoxK = 64;                       // K elements per box (128 bytes of a row)
constexpr int kWBox = kRows * kBoxK * 2;        // 16 KiB
constexpr int kXBox = kCols * kBoxK * 2;        // 2 KiB
constexpr int kBoxBytes = kWBox + kXBox;        // a multiple of 1024 (swizzle atoms)
constexpr int kThreads = 192;                   // producer, MMA and four epilogue warps
constexpr int kTmemCols = 32;                   // two 16-column accumulators
constexpr int kMaxRingSlots = 16;               // shared-memory stages
constexpr int kMaxNb = 4;                       // boxes per stage
constexpr int kMaxSplit = 16;                   // CTAs of a cluster sharing a tile

}  // namespace tc05
}  // namespace sk
