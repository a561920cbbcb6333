// pnq_split.cuh -- how the fast GEMV kernels cut a weight matrix across thread-block clusters.
//
// The rows are cut into pieces of kPieceRows rows; every cluster of C CTAs (C = 1 or 2) takes a
// contiguous run of pieces, as even as whole pieces allow, so no row is shared by two clusters.
// Inside a cluster the rows form row groups of 16 (the mma tile height; the last one may hold a
// single piece) and the K axis forms units (a fixed number of weights per row, one tensor-map
// copy wide). The items of a cluster are (unit, row group) pairs numbered unit-major; CTA r of
// the cluster takes items [r * I / C, (r + 1) * I / C), so the CTAs of a cluster stream the same
// number of bytes, each covers a few consecutive units (its x operands are built per unit), and
// every row's partial sums over the units meet in shared memory and then, across the cluster,
// through distributed shared memory -- nothing leaves the chip before the final sum.
//
// A stage is the run of consecutive items of one unit inside one block of kStageGroups row
// groups; the stages of a CTA alternate between its two consumer-warp groups by the parity of
// that block, so a row group is always handled by the same warp, whatever the unit.
#pragma once

#include <cstdint>

namespace pnq {

constexpr int kPieceRows = 8;    // rows per tensor-map copy and granularity of a cluster's rows
constexpr int kGroupRows = 16;   // rows of one mma tile
constexpr int kStageGroups = 4;  // row groups per stage block

struct Split {
    int64_t pieces;  // ceil(N / kPieceRows)
    int U;           // K units
    int ncl, C;      // clusters, CTAs per cluster

    // rows of cluster c: pieces [p0, p1)
    __host__ __device__ int64_t piece0(int c) const { return static_cast<int64_t>(c) * pieces / ncl; }
    struct Cta {
        int64_t row0;  // first row of the cluster
        int rows;      // rows of the cluster (pieces * 8; the last cluster may run past N)
        int Rg;        // row groups of the cluster
        int64_t i0, i1;  // this CTA's items (unit-major: item = u * Rg + g)
    };
    __host__ __device__ Cta cta(int block) const {
        Cta t;
        const int c = block / C, r = block % C;
        const int64_t p0 = piece0(c), p1 = piece0(c + 1);
        t.row0 = p0 * kPieceRows;
        t.rows = static_cast<int>((p1 - p0) * kPieceRows);
        t.Rg = (t.rows + kGroupRows - 1) / kGroupRows;
        const int64_t I = static_cast<int64_t>(t.Rg) * U;
        t.i0 = r * I / C;
        t.i1 = (r + 1) * I / C;
        return t;
    }
};

// One stage: unit u, row groups [g0, g1) of the cluster, stage block b = g0 / kStageGroups.
struct Stage {
    int u, g0, g1, blk;
};

// Walks the stages of one CTA in order (32-bit and incremental: no division per stage; the
// host only accepts shapes whose items per cluster fit in 32 bits).
struct StageWalk {
    int Rg, u, g, left;  // next position (unit u, row group g) and items left
    __host__ __device__ explicit StageWalk(const Split::Cta& t)
        : Rg(t.Rg), u(static_cast<int>(t.i0 / t.Rg)), g(static_cast<int>(t.i0 % t.Rg)),
          left(static_cast<int>(t.i1 - t.i0)) {}
    __host__ __device__ bool next(Stage& s) {
        if (left <= 0) return false;
        s.u = u;
        s.g0 = g;
        s.blk = g / kStageGroups;
        const int gend = (s.blk + 1) * kStageGroups < Rg ? (s.blk + 1) * kStageGroups : Rg;
        const int n = gend - g < left ? gend - g : left;
        s.g1 = g + n;
        left -= n;
        g += n;
        if (g == Rg) {
            g = 0;
            ++u;
        }
        return true;
    }
};

}  // namespace pnq
