// bounds.cuh -- index checks of the debug-bounds build.
//
// Built with -DBI_DEBUG_BOUNDS (libbi_gemm_debug.so), the GEMM and the
// decode-attention kernels check their tile coordinates and their shared-
// memory, tensor-memory and workspace indices against the bounds of what they
// address, before each access.  A failed check skips the access (it never
// traps: the GPU and the context stay usable), records BI_ERR_DEBUG_BOUNDS in
// the device status word, and, for the first failure, the check's number and
// the offending value in the detail word beside it; a skipped copy leaves its
// barrier short, so the kernel then gives up through its bounded waits.  In
// the ordinary build every check is the constant true and costs nothing.
#pragma once

#include <cstdint>

#include "bi_gemm.h"

namespace bi {

// Check numbers recorded in the detail word (bits 48..63; the value in bits 0..47).
enum BoundsCheck : uint32_t {
  kChkWStage = 1,      // W ring stage index within the W stages
  kChkXStage = 2,      // X ring stage index within the X stages
  kChkKTile = 3,       // K tile of a copy within [0, k_tiles + copy tiles)
  kChkWRow = 4,        // W row of a copy within the tile grid
  kChkXRow = 5,        // X row of a copy within the tile grid
  kChkTmemCol = 6,     // accumulator columns within the tensor-memory allocation
  kChkFoldPart = 7,    // GLOBAL fold: partial index within the workspace's partials
  kChkFoldTile = 8,    // GLOBAL fold: tile counter index within the counters
  kChkClusterPart = 9, // CLUSTER fold: DSMEM partial offset within the partial tile
  kChkAttnStage = 10,  // decode attention: stage within the CTA's pool
  kChkAttnRecord = 11, // decode attention: split record within the records
  kChkAttnItem = 12,   // decode attention: item's request, split or head within range
};

// True when `ok`.  Debug-bounds build: a false `ok` records the failure
// (status word at `status`, detail word at status + 2) and returns false, so
// that the caller skips the access.
__device__ __forceinline__ bool bounds_ok(bool ok, int* status, uint32_t check, uint64_t value) {
#ifdef BI_DEBUG_BOUNDS
  if (!ok) {
    if (status != nullptr && atomicCAS(status, 0, (int)BI_ERR_DEBUG_BOUNDS) == 0)
      *reinterpret_cast<unsigned long long*>(status + 2) =
          ((unsigned long long)check << 48) | (value & 0xFFFFFFFFFFFFull);
    return false;
  }
  return true;
#else
  (void)status;
  (void)check;
  (void)value;
  return true;
#endif
}

}  // namespace bi
