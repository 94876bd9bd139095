// Tile scheduler arithmetic shared by the host planner and the kernel.
//
// Rasterization: "4. Pipeline Abstraction and Two Consumer Warp Groups",
// section "Tile Rasterization".  The N axis of the tile grid is cut into
// groups of `width` columns; tiles inside a group are numbered row-major
// (N fastest), group after group, and the last group is narrower when
// tiles_n is not a multiple of `width`, so the map stays a bijection of
// [0, tiles_m * tiles_n).  Tiles with neighbouring ids -- the ones a wave
// of persistent CTAs works on at the same time -- then share a few B
// column strips and a few A row strips, which keeps them in L2.
//
// Division by run-time-constant divisors uses the multiply-high-and-shift
// method of Granlund and Montgomery ("Division by Invariant Integers using
// Multiplication", PLDI 1994, section 4): for a 32-bit divisor d >= 1 take
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1; then for every
// 32-bit n, floor(n / d) = (umulhi(m, n) + n) >> l, the sum taken in 64 bits.
// The same section of "4. Pipeline Abstraction..." motivates it: the group
// size is a per-launch constant, not a compile-time one.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__ __forceinline__
#else
#define GEMM_HD inline
#endif

namespace gemm_f16 {

struct FastDiv {
    uint32_t d;      // divisor (>= 1)
    uint32_t mul;    // magic multiplier
    uint32_t shift;  // l = ceil(log2 d)
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while (l < 32 && (uint64_t(1) << l) < d) ++l;
    f.shift = l;
    uint64_t numer = (uint64_t(1) << 32) * ((uint64_t(1) << l) - d);
    f.mul = uint32_t(numer / d + 1);
    return f;
}

GEMM_HD uint32_t umulhi32(uint32_t a, uint32_t b)
{
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return uint32_t((uint64_t(a) * uint64_t(b)) >> 32);
#endif
}

GEMM_HD uint32_t fast_div(const FastDiv &f, uint32_t n)
{
    uint64_t t = uint64_t(umulhi32(f.mul, n)) + uint64_t(n);
    return uint32_t(t >> f.shift);
}

// The raster of one launch: divisors precomputed on the host.
struct Raster {
    uint32_t tiles_m;
    uint32_t tiles_n;
    uint32_t width;        // N-columns per full group
    uint32_t last_width;   // width of the final group (1..width)
    uint32_t full_groups;  // number of groups of `width` columns
    FastDiv by_group;      // divide by width * tiles_m
    FastDiv by_width;      // divide by width
    FastDiv by_last;       // divide by last_width
};

inline Raster make_raster(uint32_t tiles_m, uint32_t tiles_n, uint32_t width)
{
    Raster r;
    if (width < 1) width = 1;
    if (width > tiles_n) width = tiles_n;
    r.tiles_m = tiles_m;
    r.tiles_n = tiles_n;
    r.width = width;
    r.full_groups = tiles_n / width;
    uint32_t rem = tiles_n - r.full_groups * width;
    r.last_width = rem ? rem : width;
    r.by_group = make_fastdiv(width * tiles_m);
    r.by_width = make_fastdiv(width);
    r.by_last = make_fastdiv(r.last_width);
    return r;
}

// tile id -> (m_block, n_block)
GEMM_HD void raster_coord(const Raster &r, uint32_t tile, uint32_t &m_blk, uint32_t &n_blk)
{
    uint32_t g = fast_div(r.by_group, tile);
    uint32_t in_group = tile - g * r.by_group.d;
    uint32_t n0 = g * r.width;
    const FastDiv &w = (g < r.full_groups) ? r.by_width : r.by_last;
    uint32_t m = fast_div(w, in_group);
    m_blk = m;
    n_blk = n0 + (in_group - m * w.d);
}

}  // namespace gemm_f16
