// ls_tmap.h -- host helper: build TMA tensor maps (cuTensorMapEncodeTiled, fetched from
// the driver through the runtime so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

// bf16 tensor of `rank` dims (innermost first) with byte strides of dims 1.., a box of
// `box` elements, 128-byte swizzle, zero fill out of bounds.  Returns false on failure.
bool ls_make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box);
