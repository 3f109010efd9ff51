// Resident path (k_resident.cu): configuration and launchers.  Not part of
// the public C ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace muon {

// Largest min dim and columns per CTA the resident kernel takes: the iterate
// is padded to 128 rows, and a CTA's slice of it (128 x 512 16-bit values,
// 128 KB) shares the 227 KB of shared memory with A / Q (32 KB) and the fp32
// partial Gram matrix (64 KB).
constexpr int32_t kResidentMaxM = 128;
constexpr int32_t kResidentMaxWidth = 512;
// Clusters of up to 8 CTAs (the portable size), hence n <= 8 x 512.
constexpr int32_t kResidentMaxCluster = 8;

struct ResidentCfg {
  int32_t cluster;  // CTAs per member (1, 2, 4 or 8)
  int32_t width;    // columns of the wide iterate owned by one CTA (a multiple of 64)
};

// The configuration for a group of min dim m and max dim n, a function of
// (m, n) only; false when the shape does not fit (m > 128 or n > 4096).
// The smallest cluster whose CTAs hold at most 512 columns each: fewer CTAs
// per member means fewer cluster barriers and exchanges per step for the
// same bytes.
bool resident_config(int64_t m, int64_t n, ResidentCfg* cfg);
cudaError_t prepare_resident(int ns_type);  // function attributes
cudaError_t launch_resident(const KArgs& a, const ResidentCfg& cfg, cudaStream_t s);

}  // namespace muon
