// Launch defaults of the decode kernels, shared by the launcher
// (paged_attn_decode.cu) and the host-side schedule (decode_schedule.cpp), so
// that a schedule built on the host matches what the launch does.
#pragma once

namespace pagedkv {

// Split-K partition length when the caller passes 0.
constexpr int kDefaultPartition = 512;

// Largest heads_per_cta a decode launch accepts.
constexpr int kMaxHeadsPerCta = 8;

// Two heads per block and two stages keep each block at ~32 KB of shared
// memory, so six blocks (twelve consumer warps) share an SM: measured on GB300,
// more resident consumer warps beat deeper pipelines, because each warp's
// per-chunk work is a chain of dependent shuffles and exponentials.
inline int auto_heads_per_cta(int num_heads) { return num_heads % 2 == 0 ? 2 : 1; }

}  // namespace pagedkv
