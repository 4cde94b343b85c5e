// tma.h -- host helpers that describe strided [batch][head][row][element]
// 16-bit tensors to the TMA unit (cuTensorMapEncodeTiled, reached through the
// runtime's driver entry point so the library needs no libcuda link).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace attn {

// 4-D map over [batch][head][row][element] with a {64 elements, box_rows rows}
// box and 128-byte swizzle.  Returns false when TMA cannot describe the view
// (the caller then takes another path).
bool tma_map_bhsd(CUtensorMap* m, const void* base, int dtype, int D, int rows, int heads, int batch,
                  const Layout& l, int box_rows);

// True when the view starts on a 16-byte boundary and every stride whose
// extent exceeds 1 is a positive multiple of 16 bytes.
bool tma_layout_ok(const void* base, const Layout& l, int rows, int heads, int batch);
// The same for elements of `es` bytes.
bool tma_layout_ok_es(const void* base, const Layout& l, int rows, int heads, int batch, int es);

// 4-D map over an 8-bit [batch][head][row][element] view (D elements a row)
// with a {D bytes, box_rows rows} box and 128-byte swizzle (D <= 128).
bool tma_map_bhsd_u8(CUtensorMap* m, const void* base, int D, int rows, int heads, int batch, const Layout& l,
                     int box_rows);

}  // namespace attn
