// Tile shapes of the single-pass scan, shared by the launchers and the host
// dispatcher so that both agree on the tile size.
#pragma once
#include "sc_launch.h"

namespace scg {

enum { SHAPE_LOAD_DIRECT = 0, SHAPE_LOAD_XPOSE = 1 };

// uint32 sum: variant 0 is the default; the others exist for on-GPU comparison.
constexpr ScanShape kShapeSumU32[kNumSumU32Variants] = {
    {256, 16, SHAPE_LOAD_XPOSE, 1, 1, 0},   // 4096-element tiles, coalesced loads + smem transpose
    {256, 16, SHAPE_LOAD_DIRECT, 1, 1, 0},  // 4096-element tiles, per-thread 16-byte loads
    {256, 32, SHAPE_LOAD_XPOSE, 1, 1, 0},   // 8192-element tiles
    {512, 16, SHAPE_LOAD_XPOSE, 1, 1, 0},   // 8192-element tiles, 16 warps
    {128, 32, SHAPE_LOAD_XPOSE, 1, 1, 0},   // 4096-element tiles, 4 warps
    {256, 16, SHAPE_LOAD_XPOSE, 4, 1, 0},   // 4096, look-back 128 tiles per round trip
    {256, 32, SHAPE_LOAD_XPOSE, 4, 1, 0},   // 8192, look-back 128
    {512, 16, SHAPE_LOAD_XPOSE, 4, 1, 0},   // 8192, 16 warps, look-back 128
    {256, 16, SHAPE_LOAD_XPOSE, 4, 8, 0},   // 4096, look-back 128, 8 CTAs/SM (<= 32 registers)
    {512, 32, SHAPE_LOAD_XPOSE, 4, 1, 0},   // 16384-element tiles, look-back 128
    {256, 16, SHAPE_LOAD_XPOSE, 4, 6, 0},   // 4096, look-back 128, 6 CTAs/SM
    {256, 16, SHAPE_LOAD_XPOSE, 1, 6, 0},   // 4096, look-back 32, 6 CTAs/SM
    {256, 16, SHAPE_LOAD_XPOSE, 1, 1, 1},   // variant 0 with phase timers
    {128, 32, SHAPE_LOAD_XPOSE, 1, 1, 1},   // variant 4 with phase timers
    {256, 16, SHAPE_LOAD_XPOSE, 4, 8, 1},   // variant 8 with phase timers
};
constexpr ScanShape kShapeSumF32 = {256, 16, SHAPE_LOAD_XPOSE, 1, 1, 0};
constexpr ScanShape kShapeMaxI32 = {256, 16, SHAPE_LOAD_XPOSE, 1, 1, 0};
constexpr ScanShape kShapeAffine = {256, 8, SHAPE_LOAD_XPOSE, 1, 1, 0};  // 8-byte elements
// the operators run through launch_scan_extra, by element size
constexpr ScanShape kShapeExtra4 = {256, 16, SHAPE_LOAD_XPOSE, 1, 1, 0};
constexpr ScanShape kShapeExtra8 = {256, 8, SHAPE_LOAD_XPOSE, 1, 1, 0};

}  // namespace scg
