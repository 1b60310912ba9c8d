// Tile shapes of the single-pass scan, shared by the launchers and the host
// dispatcher so that both agree on the tile size.
#pragma once
#include "sc_launch.h"

namespace scg {

enum { SHAPE_LOAD_DIRECT = 0, SHAPE_LOAD_XPOSE = 1 };

// uint32 sum: variant 0 is the default; the others exist for on-GPU comparison.
constexpr ScanShape kShapeSumU32[kNumSumU32Variants] = {
    {256, 16, SHAPE_LOAD_XPOSE},   // 4096-element tiles, coalesced loads + smem transpose
    {256, 16, SHAPE_LOAD_DIRECT},  // 4096-element tiles, per-thread 16-byte loads
    {256, 32, SHAPE_LOAD_XPOSE},   // 8192-element tiles
    {512, 16, SHAPE_LOAD_XPOSE},   // 8192-element tiles, 16 warps
    {128, 32, SHAPE_LOAD_XPOSE},   // 4096-element tiles, 4 warps
};
constexpr ScanShape kShapeSumF32 = {256, 16, SHAPE_LOAD_XPOSE};
constexpr ScanShape kShapeMaxI32 = {256, 16, SHAPE_LOAD_XPOSE};
constexpr ScanShape kShapeAffine = {256, 8, SHAPE_LOAD_XPOSE};  // 8-byte elements

}  // namespace scg
