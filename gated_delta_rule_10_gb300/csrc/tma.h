// Host-side creation of TMA tensor maps (driver entry point looked up at run
// time, so the library needs no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

// A [B, T, H, D] bf16 tensor (D fastest) seen as a 4-D TMA map with a box of
// 64 channels x 1 head x 64 tokens x 1 batch and the 128-byte swizzle, so each
// load of one (channel block, head, chunk, batch) lands as an 8 KB operand block
// in the layout of tc.cuh. Tokens past T read as zeros. Returns false when the
// driver refuses the description.
bool make_bthd_tmap(CUtensorMap* map, const void* base, int B, int T, int H, int D);

}  // namespace gdr
