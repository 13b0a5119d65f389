// Tensor maps of the MLA decode kernels (q and the paged latent cache).
#pragma once

#include <cuda.h>

#include <cstdint>

namespace pda {

// With S = dqk / 64 sub-tiles per record (9 for 576, 5 for 320):
// q [rows, dqk]: dims (d mod 64, row, d / 64), box (64, n, S) -> S [n][64] sub-tiles.
// kv [blocks, 64, dqk]: dims (d mod 64, slot, d / 64, block), box (64, 64, S, 1) ->
// S [64][64] sub-tiles per page. Both 16-bit with the 128-byte swizzle. Returns false when
// the driver's encoder is unavailable or rejects the maps.
bool encode_mla_maps(CUtensorMap* tq, CUtensorMap* tkv, const void* q, int64_t rows, int n,
                     const void* kv, int64_t num_blocks, bool bf16, int dqk);

}  // namespace pda
