// pnq_streamk.cuh -- the work split shared by the tensor-core GEMV kernels (PN and NVFP4).
//
// Items are 128 weight rows x one K unit; a persistent grid takes equal contiguous shares of
// them (stream-K). Consumer warps leave each finished tile's row sums in shared memory; a reducer
// warp writes a tile the CTA covered whole straight to Y, and otherwise stores the CTA's share of
// it in a workspace slot; at the end the CTA counts its shares (one atomic each) and the CTA
// that completes a tile sums its slots in unit order (so results do not depend on timing).
#pragma once

#include <cstdint>

#include "pnq_device.cuh"

namespace pnq {
namespace {

constexpr int kTileRows = 128;        // rows per item
constexpr int kPartPitch = 132;       // floats per (half, buffer, m) row-sum vector in shared memory
constexpr int kMaxStages = 8;
constexpr unsigned kStaticWeights = 1u;
constexpr size_t kSmemLimit = 227u * 1024u;

// Item numbering. Tile-major (item = t * U + u): a CTA's share covers one or two row tiles and
// at most U units, and it accumulates a tile over consecutive items. Unit-major (item = u * T + t):
// a CTA's share touches at most a few units (for operands that would not fit otherwise). CTA c
// of G takes items [c * items / G, (c + 1) * items / G).
struct Sched {
    int items;  // T * U < 2^31 (checked by the host)
    int T, U, G, tile_major;
    __host__ __device__ int tile_of(int i) const { return tile_major ? i / U : i % T; }
    __host__ __device__ int unit_of(int i) const { return tile_major ? i % U : i / T; }
    __host__ __device__ int item(int t, int u) const { return tile_major ? t * U + u : u * T + t; }
    __host__ __device__ int first(int c) const { return static_cast<int>(static_cast<long long>(c) * items / G); }
    __host__ __device__ int owner(int i) const {
        return static_cast<int>((static_cast<long long>(i + 1) * G - 1) / items);
    }
    // A share is a run of consecutive items of one CTA within a tile. Tile-major (or T = 1):
    // the items of tile t are consecutive, a share starts at unit 0 and at the first item of
    // every CTA that begins inside the tile. Unit-major: every unit is a share of its own.
    __host__ __device__ bool consecutive() const { return tile_major || T == 1; }
    __host__ __device__ int shares(int t) const {
        if (!consecutive()) return U;
        const int a0 = item(t, 0);
        return owner(a0 + U - 1) - owner(a0) + 1;
    }
    // units a CTA's share touches (a cyclic range starting at unit_of(first item))
    __host__ __device__ int span(int i0, int i1) const {
        if (i1 <= i0) return 0;
        if (tile_major) return i1 - i0 < U ? i1 - i0 : U;
        return unit_of(i1 - 1) - unit_of(i0) + 1;
    }
};

// Kernel parameters the loops read, copied once into registers (parameters reached through a
// pointer would be reloaded after every barrier).
struct Ctx {
    Sched sc;
    const void* X;  // activations: fp32 (PN) or bf16 (NVFP4)
    float* Y;
    float* ws;
    uint32_t* cnt;
    int* err;
    int N, K, M, NS, x_stage, xpitch;
    unsigned flags;
};

// Next item of a share: (t, u) in the share's order, without divisions.
__device__ __forceinline__ void next_item(const Sched& sc, int& t, int& u) {
    if (sc.tile_major) {
        if (++u == sc.U) {
            u = 0;
            ++t;
        }
    } else if (++t == sc.T) {
        t = 0;
        ++u;
    }
}

// Y rows t*128 + 4*lane .. + 3 of activation row m.
__device__ __forceinline__ void put_y(const Ctx& a, int t, int m, int lane, float4 v) {
    const int row = t * kTileRows + 4 * lane;
    float* y = a.Y + static_cast<size_t>(m) * a.N;
    if (row + 0 < a.N) y[row + 0] = v.x;
    if (row + 1 < a.N) y[row + 1] = v.y;
    if (row + 2 < a.N) y[row + 2] = v.z;
    if (row + 3 < a.N) y[row + 3] = v.w;
}

// Reducer side of one share of tile t (consecutive items of this CTA, units u_first ..
// u_first+n-1): add the two halves; a whole tile goes to Y, a part to its workspace slot (it is
// counted later). Returns true for a part.
template <int MAXM, class SM>
__device__ __forceinline__ bool reduce_share(const Ctx& a, const SM& sm, int buf, int t, int u_first, int n_units,
                                             int lane) {
    const Sched& sc = a.sc;
    // the two halves' row sums into registers; the buffer goes back to the consumers at once
    const float* part = sm.part();
    float4 v[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        if (m < a.M) {
            const float4 p0 = reinterpret_cast<const float4*>(part + ((0 * 2 + buf) * a.M + m) * kPartPitch)[lane];
            const float4 p1 = reinterpret_cast<const float4*>(part + ((1 * 2 + buf) * a.M + m) * kPartPitch)[lane];
            v[m] = make_float4(p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.part_free(buf));
    if (n_units == sc.U) {
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
            if (m < a.M) put_y(a, t, m, lane, v[m]);
        return false;
    }
    float* slot = a.ws + (static_cast<size_t>(t) * sc.U + u_first) * a.M * kTileRows;
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
        if (m < a.M) __stcg(reinterpret_cast<float4*>(slot + m * kTileRows) + lane, v[m]);
    return true;
}

// Count the np partial shares of this CTA (tiles in pending[]) after their slots were stored:
// the ones that complete their tile are appended to finish[] (n_finish[0] entries). One warp.
template <class SM>
__device__ __forceinline__ void count_shares(const Ctx& a, const SM& sm, int np, int lane) {
    __threadfence();  // the slots are visible before they are counted
    __syncwarp();
    int* pend = sm.pending();
    int* fin = sm.finish();
    for (int k0 = 0; k0 < np; k0 += 32) {
        const int k = k0 + lane;
        bool last = false;
        int t = 0;
        if (k < np) {
            t = pend[k];
            last = atomicAdd(a.cnt + t, 1u) == static_cast<unsigned>(a.sc.shares(t) - 1);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, last);
        const int base = *sm.n_finish();
        if (last) fin[base + __popc(mask & ((1u << lane) - 1u))] = t;
        __syncwarp();
        if (lane == 0) *sm.n_finish() = base + __popc(mask);
        __syncwarp();
    }
    __threadfence();  // what the other CTAs stored before counting is seen by the finishers
}

// Sum the shares of tile t in unit order into Y and clear its counter (one warp).
__device__ __forceinline__ void finish_tile(const Ctx& a, int t, int lane) {
    const Sched& sc = a.sc;
    for (int m = 0; m < a.M; ++m) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        auto add_slot = [&](int u) {
            const float* slot = a.ws + ((static_cast<size_t>(t) * sc.U + u) * a.M + m) * kTileRows;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(slot) + lane);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        };
        if (sc.consecutive()) {
            const int a0 = sc.item(t, 0);
            add_slot(0);
            for (int c = sc.owner(a0) + 1; c <= sc.owner(a0 + sc.U - 1); ++c) add_slot(sc.first(c) - a0);
        } else {
            for (int u = 0; u < sc.U; ++u) add_slot(u);
        }
        put_y(a, t, m, lane, acc);
    }
    __syncwarp();
    if (lane == 0) a.cnt[t] = 0u;  // ready for the next launch
}

// ---- host ----------------------------------------------------------------------------------

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }


}  // namespace
}  // namespace pnq
