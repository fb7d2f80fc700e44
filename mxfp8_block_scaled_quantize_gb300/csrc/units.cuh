// A warp's walk over the units u0, u0 + stride, u0 + 2 stride, ... of a grid
// laid out as bands of `cols` units, kept as (band, col) so that a step costs
// an add and a compare instead of a 64-bit division.
#pragma once
#include <cstdint>

namespace temx {

struct UnitWalk {
    int32_t dband, dcol, cols;
    __device__ __forceinline__ UnitWalk(int64_t stride, int64_t ncols)
        : dband(int32_t(stride / ncols)), dcol(int32_t(stride % ncols)), cols(int32_t(ncols)) {}
    __device__ __forceinline__ void start(int64_t u0, int32_t& band, int32_t& col) const {
        band = int32_t(u0 / cols);
        col = int32_t(u0 % cols);
    }
    __device__ __forceinline__ void step(int32_t& band, int32_t& col) const {
        col += dcol;
        band += dband;
        if (col >= cols) {
            col -= cols;
            ++band;
        }
    }
};

}  // namespace temx
