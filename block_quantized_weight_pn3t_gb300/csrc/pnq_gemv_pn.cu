// pnq_gemv_pn.cu -- PN (pn3t / pn4t) GEMV on the tensor cores with mma.sync, sm_103a (fast path).
//
// Computes Y[m][n] = sum_k w[n][k] x[m][k] for 1 <= M <= 16, with w = d * (n - z) decoded in
// registers from the 34-byte blocks of the "PN weight format" page (sections Block layout and
// Value) just before the multiply. A K unit is 8 blocks (272 bytes of a row). Two pipelines:
//   - the row stream (M <= 8; below): clusters of 1..8 CTAs own rows, each CTA a share of their
//     K units; stages of 16 rows (or of a K segment of 16 rows) arrive by one 1-D bulk copy per
//     row, and the B operands of the CTA's units stay in shared memory;
//   - the cluster strip pipeline (pnq_cluster.cuh, with this file's PnMma policy): 2-D tensor-map
//     copies of 8- and 64-row strips of a unit, clusters of one or two CTAs sharing row tiles and
//     summing through distributed shared memory; it takes M = 9..16 and the M <= 8 shapes whose B
//     operands do not fit beside a row-stream ring.
//
// Decode and multiply. A 32-bit word of a block holds two codes at the same shift in its two
// 16-bit halves; masking out one such pair leaves in each half the exact fp16 subnormal
// n * 2^-24 * 8^j (pn3t; 16^j for pn4t, j the pair's position, the word shifted right by 9 / 8
// bits first for the pairs past fp16's mantissa): one AND per two weights gives an mma A
// register. Lane (g, c) of a warp uses words c and c + 4 of rows g and g + 8 (m16n8k16: a0/a1 =
// word c of rows g / g + 8, a2/a3 = word c + 4). Odd blocks' words are 4-byte aligned in a
// 16-byte aligned row; even blocks are read as the aligned words that pair the high half of word
// i with the low half of word i + 1 (the k order inside a block is free as long as B follows it),
// and the one pair that straddles the block end (word 7 high, word 0 low) is joined with a PRMT.
// Four blocks' mma chains are interleaved step by step (four accumulations in flight per warp).
//
// B operand (per K unit and activation row m): x * 2^sigma * 2^-(shift of the pair), sigma so that
// max |x| * 2^sigma over the unit lies in [2^14, 2^15), split into fp16 hi (the leading 11 bits)
// and lo (the remainder, rounded) in mma columns 2m and 2m + 1. A block's two column sums added
// give sum_k c_k x_k * 2^(sigma - 24); minus Z = z * 2^(sigma - 24) * (sum of the block's x) and
// times d that is the block's share of the row sum, and each unit's sums are scaled by
// 2^(24 - sigma) into the row partials.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pnq_cluster.cuh"

namespace pnq {
namespace {

constexpr int kUnitBlocks = 8;                           // blocks per K unit
constexpr int kUnitBytes = kUnitBlocks * kBlockBytes;    // 272 bytes of a row per unit
constexpr int kUnitU32 = kUnitBytes / 4;                 // 68
constexpr int kStageBytes = kStageRows * kUnitBytes;     // 17408
constexpr int kPieceBytes = kPieceRows * kUnitBytes;     // 2176 (one copy)

// LR = lanes whose B records are stored (32, or the 8M lanes of the live columns when one n8 tile
// is only partly used: the other lanes read a live column's record).
template <int TYPE, int NT, int LR = 32>
struct Cfg {
    using F = PnFmt<TYPE>;
    static constexpr int STEPS = F::PAIRS;
    static constexpr int UK = kUnitBlocks * F::BLK;     // weights of a row per unit (640 / 512)
    // B records of one (block, n8 tile): STEPS / 2 pairs of steps as 16-byte lane records, then
    // the odd last step as 8-byte lane records
    static constexpr int PAIR = LR * 16;                // bytes of one pair-of-steps record group
    static constexpr int PB = (STEPS / 2) * PAIR + (STEPS & 1) * LR * 8;
    static constexpr int REC = kUnitBlocks * NT * PB;   // bytes of one unit's B operands
    static constexpr int SH = (TYPE == kTypePn3t) ? 9 : 8;
    static constexpr int JS = (TYPE == kTypePn3t) ? 3 : 2;  // pairs below the shift
};

// fp16 in the low / high half of a word -> fp32
__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w))); }
__device__ __forceinline__ float half_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Masked pair J of a word (w) or of the word shifted right by SH (s).
template <int TYPE, int J>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t s) {
    if constexpr (TYPE == kTypePn3t) {
        if constexpr (J < 3) return w & (0x00070007u << (3 * J));
        else return s & (0x00070007u << (3 * (J - 3)));
    } else {
        if constexpr (J < 2) return w & (0x000F000Fu << (4 * J));
        else return s & (0x000F000Fu << (4 * (J - 2)));
    }
}

// Element of the block held by half h (0 = low) of decode register r (0: word c, 1: word c + 4)
// at pair j, for lane column c: odd blocks read the words themselves; even blocks read the
// aligned word that pairs the high half of word i (odd codes) with the low half of word i + 1
// (even codes), i = c or c + 4, and word 7 wraps to word 0.
__device__ __forceinline__ int pn_elem(int cpw, bool odd, int c, int r, int j, int h) {
    const int i = c + 4 * r;
    if (odd) return cpw * i + 2 * j + h;
    return h ? cpw * ((i + 1) & 7) + 2 * j : cpw * i + 2 * j + 1;
}

// B operands of one K unit for activation row m (one builder warp): sigma from the row's largest
// |x| over the unit, the hi / lo lane records of every (block, lane column, pair) and the blocks'
// zero-point terms (zb[block * ZS + m]: ZS activation rows per block); xr = the unit's x row in
// shared memory.
template <int TYPE, int NT, int LR = 32, int ZS = 16>
__device__ __forceinline__ void build_row(uint8_t* rec, float* zb, float* so, const float* xr, int m, int lane) {
    using C = Cfg<TYPE, NT, LR>;
    using F = PnFmt<TYPE>;
    constexpr int STEPS = C::STEPS, UK = C::UK;
    uint32_t mx = 0;  // a non-negative float's bits order like its value
#pragma unroll
    for (int q = lane; q < UK / 4; q += 32) {
        const float4 v = reinterpret_cast<const float4*>(xr)[q];
        mx = max(mx, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                         max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int E = static_cast<int>(mx >> 23);
    int sg = (mx == 0 || E >= 255) ? 0 : 141 - E;  // max |x| < 2^(E - 126)
    sg = min(100, max(-100, sg));
    const int t = m >> 2;                            // n8 tile of columns 2m, 2m + 1
    const int lh = (((2 * m) & 7) << 2), ll = (((2 * m + 1) & 7) << 2);
    // tasks (block, lane column c, pair j)
    constexpr int TASKS = kUnitBlocks * 4 * STEPS;
#pragma unroll
    for (int k0 = 0; k0 < TASKS; k0 += 32) {
        const int k = k0 + lane;
        if (TASKS % 32 == 0 || k < TASKS) {
            const int blk = k / (4 * STEPS), r0 = k - blk * 4 * STEPS;
            const int c = r0 / STEPS, j = r0 - c * STEPS;
            const bool odd = blk & 1;
            const float* xb = xr + blk * F::BLK;
            const float sc = exp2i(sg - (F::BITS * (j % C::JS)));
            uint32_t hi[2], lo[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint64_t xp = f32x2_pack(xb[pn_elem(F::CPW, odd, c, r, j, 0)], xb[pn_elem(F::CPW, odd, c, r, j, 1)]);
                uint64_t hp, lp;
                split11x2(f32x2_mul(xp, f32x2_pack(sc, sc)), hp, lp);
                float h0, h1, l0, l1;
                f32x2_unpack(hp, h0, h1);
                f32x2_unpack(lp, l0, l1);
                hi[r] = f32x2_to_f16x2(h0, h1);  // exact
                lo[r] = f32x2_to_f16x2(l0, l1);
            }
            uint8_t* tb = rec + (blk * NT + t) * C::PB;
            if (j < 2 * (STEPS / 2)) {
                uint8_t* p = tb + (j >> 1) * C::PAIR + (j & 1) * 8;
                *reinterpret_cast<uint2*>(p + (lh + c) * 16) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2*>(p + (ll + c) * 16) = make_uint2(lo[0], lo[1]);
            } else {
                uint8_t* p = tb + (STEPS / 2) * C::PAIR;
                *reinterpret_cast<uint2*>(p + (lh + c) * 8) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2*>(p + (ll + c) * 8) = make_uint2(lo[0], lo[1]);
            }
        }
    }
    // zero-point terms: lane = 4 * block + quarter sums a quarter of the block, starting at its
    // element (lane mod QN) and wrapping around (the lanes' quarters are QN floats apart, so in
    // element order the lanes of a load would share a few banks; rotated, no bank serves more
    // than two of them)
    {
        const int blk = lane >> 2, qt = lane & 3;
        constexpr int QN = F::BLK / 4;
        const float* xq = xr + blk * F::BLK + qt * QN;
        float s = 0.0f;
        int e = lane % QN;
#pragma unroll
        for (int t = 0; t < QN; ++t) {
            s += xq[e];
            e = (e == QN - 1) ? 0 : e + 1;
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        // Z = z * sum over the block of 2^-24 * 2^shift * B = z * 2^(sigma - 24) * (sum of x)
        if (qt == 0) zb[blk * ZS + m] = static_cast<float>(F::Z) * s * exp2i(sg - 24);
    }
    if (lane == 0) so[m] = exp2i(24 - sg);  // undoes sigma and the 2^-24 of the codes
}

// NBK consecutive blocks B0 .. B0 + NBK - 1 (compile time, B0 even) of a row group: decode,
// multiply, fold d * (c - Z) into acc[t][h] (rows g, g + 8 of the group; column pair of
// activation row 4t + c). The blocks' mma chains are interleaved step by step, so a warp keeps
// NBK independent accumulations in flight. Every shared-memory load is a 32-bit shared address
// in a register plus a compile-time offset:
//   srow[h] / srow_c[h]: row g (h = 0) and row g + 8 (h = 1) of the group at the K unit's first
//   byte (srow_c = srow + 4c, lane column c's words), so any row stride works;
//   srec[t]: the B records of tile t at the lane's record (lanes of columns past 2M read a live
//   column's record: their sums are never used), srec_h[t] the same for 8-byte records;
//   szb[t]: the zero-point term of the lane's activation row (clamped the same way) in a table of
//   ZS activation rows per block.
template <int TYPE, int NT, int B0, int NBK, int LR = 32, int ZS = 16>
__device__ __forceinline__ void pn_blocks(const uint32_t (&srow)[2], const uint32_t (&srow_c)[2], uint32_t sel,
                                          const uint32_t (&srec)[NT], const uint32_t (&srec_h)[NT],
                                          const uint32_t (&szb)[NT], float (&acc)[NT][2]) {
    using Cf = Cfg<TYPE, NT, LR>;
    constexpr int STEPS = Cf::STEPS;
    uint32_t ra[NBK][2], rb[NBK][2], sa[NBK][2], sb[NBK][2];
    float d[NBK][2], z[NBK][NT];
    static_for<NBK>([&](auto I) {
        constexpr int i = decltype(I)::value, B = B0 + i;
        static_for<2>([&](auto Hh) {
            constexpr int h = decltype(Hh)::value, OFF = kBlockBytes * B;
            if constexpr (B & 1) {
                ra[i][h] = ld_shared_u32<OFF + 2>(srow_c[h]);
                rb[i][h] = ld_shared_u32<OFF + 18>(srow_c[h]);
                d[i][h] = half_hi(ld_shared_u32<OFF - 2>(srow[h]));
            } else {
                const uint32_t q0 = ld_shared_u32<OFF>(srow[h]);
                ra[i][h] = ld_shared_u32<OFF + 4>(srow_c[h]);
                rb[i][h] = prmt(ld_shared_u32<OFF + 20>(srow_c[h]), q0, sel);
                d[i][h] = half_lo(q0);
            }
            sa[i][h] = ra[i][h] >> Cf::SH;
            sb[i][h] = rb[i][h] >> Cf::SH;
        });
        static_for<NT>([&](auto T) {
            constexpr int t = decltype(T)::value;
            z[i][t] = ld_shared_f32<4 * ZS * B>(szb[t]);
        });
    });
    float acc4[NBK][NT][4];
    uint4 bq[NBK][NT];  // B records of a pair of steps
    static_for<STEPS>([&](auto Jc) {
        constexpr int J = decltype(Jc)::value;
        static_for<NBK>([&](auto I) {
            constexpr int i = decltype(I)::value, B = B0 + i;
            static_for<NT>([&](auto T) {
                constexpr int t = decltype(T)::value, RT = (B * NT + t) * Cf::PB;
                if constexpr ((J & 1) == 0 && J + 1 < STEPS) {
                    bq[i][t] = ld_shared_v4<RT + (J >> 1) * Cf::PAIR>(srec[t]);
                } else if constexpr ((J & 1) == 0) {
                    const uint2 v = ld_shared_v2<RT + (STEPS / 2) * Cf::PAIR>(srec_h[t]);
                    bq[i][t].x = v.x;
                    bq[i][t].y = v.y;
                }
            });
            const uint32_t a0 = code_pair<TYPE, J>(ra[i][0], sa[i][0]);
            const uint32_t a1 = code_pair<TYPE, J>(ra[i][1], sa[i][1]);
            const uint32_t a2 = code_pair<TYPE, J>(rb[i][0], sb[i][0]);
            const uint32_t a3 = code_pair<TYPE, J>(rb[i][1], sb[i][1]);
            static_for<NT>([&](auto T) {
                constexpr int t = decltype(T)::value;
                const uint32_t b0 = (J & 1) ? bq[i][t].z : bq[i][t].x, b1 = (J & 1) ? bq[i][t].w : bq[i][t].y;
                if constexpr (J == 0)
                    mma_f16_16816_z(acc4[i][t], a0, a1, a2, a3, b0, b1);
                else
                    mma_f16_16816(acc4[i][t], a0, a1, a2, a3, b0, b1);
            });
        });
    });
#pragma unroll
    for (int i = 0; i < NBK; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(d[i][0], (acc4[i][t][0] + acc4[i][t][1]) - z[i][t], acc[t][0]);
            acc[t][1] = fmaf(d[i][1], (acc4[i][t][2] + acc4[i][t][3]) - z[i][t], acc[t][1]);
        }
}

// The PN format policy of the cluster pipeline (tensor-core multiply).
template <int TYPE, int NT>
struct PnMma {
    using C = Cfg<TYPE, NT>;
    static constexpr int MAPS = 2;  // the weights with 8-row boxes (pieces) and 64-row boxes (stages)
    struct Extra {};
    static constexpr int NB = (NT == 4) ? 3 : NT;  // builder warps (12 warps at most: 168 registers)
    static constexpr int THREADS = 32 * (kConsumerWarps + 1 + NB);
    static constexpr int MINB = (NT == 1) ? 2 : 1;  // resident CTAs per SM the registers allow
    static constexpr int UK = C::UK, X_BYTES = 4;
    static constexpr int STAGE_BYTES = kStageBytes, PIECE_TX = kPieceBytes;
    static constexpr int REC = C::REC;
    static constexpr int ZB = kUnitBlocks * 16 + 16;  // zero-point terms [block][m], then 2^(24 - sigma) [m]
    static constexpr double GROUP_S = 0.22e-6;        // one warp, one row group x one unit
    struct Lane {
        int g, c;
        uint32_t sel;
        uint32_t boff[NT], zoff[NT];  // the lane's B record offset and zero-point term offset
        __device__ Lane(int l, int M) : g(l >> 2), c(l & 3), sel((l & 3) == 3 ? 0x7610u : 0x3210u) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int gc = min(g, max(0, 2 * M - 1 - 8 * t));  // a live column of the tile
                boff[t] = static_cast<uint32_t>((4 * gc + c) * 16);
                zoff[t] = static_cast<uint32_t>(4 * min(4 * t + c, M - 1));
            }
        }
    };
    struct Acc {
        float v[NT][2];
    };
    static __device__ __forceinline__ void issue(const CUtensorMap* maps, uint32_t dst, int p, int u, int row,
                                                 uint32_t bar, uint64_t pol) {
        tma_load_2d(dst + p * kPieceBytes, &maps[0], u * kUnitU32, row, bar, pol);
    }
    static __device__ __forceinline__ void issue_stage(const CUtensorMap* maps, uint32_t dst, int u, int row,
                                                       uint32_t bar, uint64_t pol) {
        tma_load_2d(dst, &maps[1], u * kUnitU32, row, bar, pol);
    }
    static __device__ __forceinline__ void zero_half(uint8_t* stg, int lg, int lane) {
        uint32_t* zp = reinterpret_cast<uint32_t*>(stg + (lg * kGroupRows + 8) * kUnitBytes);
        for (int i = lane; i < 8 * kUnitU32; i += 32) zp[i] = 0u;
    }
    static __device__ __forceinline__ void build(uint8_t* rec, float* zb, const uint8_t* xrow, int m, const Extra&,
                                                 int lane) {
        build_row<TYPE, NT>(rec, zb, zb + kUnitBlocks * 16, reinterpret_cast<const float*>(xrow), m, lane);
    }
    static __device__ __forceinline__ void group(const uint8_t* stg, int lg, const uint8_t* recu, const float* zbu,
                                                 int, const Lane& ln, Acc& acc) {
        const uint32_t s0 = smem_addr(stg) + static_cast<uint32_t>((lg * kGroupRows + ln.g) * kUnitBytes);
        const uint32_t srow[2] = {s0, s0 + 8u * kUnitBytes};
        const uint32_t srow_c[2] = {s0 + 4u * ln.c, s0 + 8u * kUnitBytes + 4u * ln.c};
        const uint32_t rec_s = smem_addr(recu), zb_s = smem_addr(zbu);
        uint32_t srec[NT], srec_h[NT], szb[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            srec[t] = rec_s + ln.boff[t];
            srec_h[t] = rec_s + ln.boff[t] / 2;
            szb[t] = zb_s + ln.zoff[t];
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) acc.v[t][0] = acc.v[t][1] = 0.0f;
        if constexpr (NT == 1) {  // four blocks' chains interleaved
            pn_blocks<TYPE, NT, 0, 4>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
            pn_blocks<TYPE, NT, 4, 4>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
        } else if constexpr (NT == 2) {  // two blocks' chains, two tiles each
            pn_blocks<TYPE, NT, 0, 2>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
            pn_blocks<TYPE, NT, 2, 2>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
            pn_blocks<TYPE, NT, 4, 2>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
            pn_blocks<TYPE, NT, 6, 2>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
        } else {  // four tiles already give four chains
            static_for<8>([&](auto Bc) {
                pn_blocks<TYPE, NT, decltype(Bc)::value, 1>(srow, srow_c, ln.sel, srec, srec_h, szb, acc.v);
            });
        }
    }
    // rows g, g + 8 of the group, activation row 4t + c: partial += sums * 2^(24 - sigma)
    static __device__ __forceinline__ void flush(float* part, int rc, int lr, const float* zbu, int M, const Lane& ln,
                                                 const Acc& acc) {
        const float* so = zbu + kUnitBlocks * 16;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int m = 4 * t + ln.c;
            if (m < M) {
                const float f = so[m];
                float* pr = part + m * rc + lr + ln.g;
                pr[0] = fmaf(acc.v[t][0], f, pr[0]);
                pr[8] = fmaf(acc.v[t][1], f, pr[8]);
            }
        }
    }
};

// ---- row-stream path (M <= 8) ----------------------------------------------------------------------
//
// A cluster of CL CTAs (CL = 1, 2, 4 or 8, chosen by rs_cost below) owns a contiguous range of
// rows; CTA r of the cluster takes K units [r U / CL, (r + 1) U / CL) of those rows: it streams
// only those bytes of each row, builds only those units' operands from only that slice of x, and
// at the end the cluster sums the CTAs' partial rows through distributed shared memory in CTA
// order (CL = 1: nothing is summed across CTAs). M <= 4 uses one n8 tile per task (columns 2m,
// 2m + 1), M = 5..8 two (one decoded A fragment, two MMAs). A stage holds 16 rows of the CTA's
// units (a row group): sixteen 1-D bulk copies, one per row, issued by the lanes of two
// producer warps, eight rows each (copies issued from two warps stream at the full HBM rate, one
// warp's at about two thirds of it; 2-D boxes of 272-byte strips stream far slower). A stage row
// is `pitch` bytes apart: its length, padded by 16 bytes where needed so that pitch / 16 is odd,
// which puts the 32 words a warp loads at once (8 rows x 4 lane columns) in 32 different
// shared-memory banks.
//
// Whole rows (SEG = false; rows of up to 16 K units): consumer warp w owns the units u = w, w + 8,
// ..; it streams the x of its own (unit, activation row) pairs through two buffers of its own,
// builds their B operands and multiplies every row group over them, storing its per-row sums in
// its own slice of shared memory.
//
// Row segments (SEG = true; longer rows): the units of a row are cut into `nseg` segments of
// near-equal length and a stage holds one segment of a row group. All of x ([M][K] fp32) comes in
// with one bulk copy per activation row, issued by consumer warp 0 once the previous grid is done
// (loads issued one unit at a time would each wait behind every weight copy in flight on the SM);
// the consumer warps then build the B operands of all units between them, (unit, activation row)
// pairs p = w, w + 8, .. for warp w, and meet at a barrier. The (row group, unit) tasks of the
// stages are dealt to the warps in turn, so each warp gets the same number of tasks to within one
// whatever the segment lengths; a warp adds its task sums into its own slice of per-row sums.
//
// Either way the slices are summed in warp order at the end.
//
// FMA = true replaces the tensor-core decode with a CUDA-core one (the plain design the measurement
// compares against; it takes the row-segment code path, all of x staged, no B operands): lane l
// of a warp takes row l / 2 of the group and words 4 (l % 2) .. 4 (l % 2) + 3 of each block; a code
// c becomes the exact float c - z by one AND-OR into the mantissa of 1.5 * 2^23 and one
// subtraction, and M fp32 FMAs with x from shared memory follow; d scales each block's sums.
//
// The SM takes in bulk copies at about the HBM rate per SM, in issue order, so x requested after
// the producer has filled the ring would land only behind all of it. The producer therefore issues
// one stage, then waits until every consumer warp has requested its x, and fills the ring behind.
// x is read only while the operands are built, so the plan may place it in the ring's last slots
// (slot 2 or later): the producer fills those only after every consumer warp has arrived on the
// "operands built" barrier.

constexpr int kRsWarps = 8;      // consumer warps
constexpr int kRsProducers = 2;  // producer warps, rows 0..7 and 8..15 of each group
constexpr int kRsThreads = 32 * (kRsWarps + kRsProducers);
constexpr int kRsWholeUnits = 16;  // longest whole row (units); longer rows are cut into segments
constexpr int kRsMaxSeg = 32;      // segments of a row at most
constexpr int kRsZs = 4;           // activation rows of the CUDA-core decode (M <= 4)
// zero-point table of NT n8 tiles (4 NT activation rows): floats per unit, terms [block][m], then
// 2^(24 - sigma) [m]
constexpr int rs_zs(int NT) { return 4 * NT; }
constexpr int rs_zb(int NT) { return kUnitBlocks * rs_zs(NT) + rs_zs(NT); }
constexpr uint32_t kRsConsumerBar = 1;              // named barrier of the consumer warps

// Stage pitch of a row (segment) of `bytes` (a multiple of 16): the least multiple of 16 >= bytes
// whose quotient by 16 is odd.
constexpr int rs_pitch(int bytes) { return ((bytes / 16) & 1) ? bytes : bytes + 16; }

struct RsArgs {
    const uint8_t* W;
    const float* X;
    float* Y;
    int* err;
    int N, K, M, U, G, S;  // G clusters of CL CTAs, S stages
    int CL;                // CTAs of a cluster: CTA r of a cluster takes K units [r U / CL, (r + 1) U / CL) of its rows
    int nseg;              // segments of a row (units [j U / nseg, (j + 1) U / nseg) for segment j)
    int row_bytes, pitch;  // a weight row in HBM; a whole row's stride in a stage
    int rows_pad;          // partial rows per (warp, activation row), >= any CTA's rows
    unsigned flags;
    uint32_t off_rec, off_zb, off_x, off_part, off_stage, stage_bytes;
    int x_slot0;  // first ring slot that holds x until the operands are built (S: x has its own region)
    int x_ahead;  // weight stages issued before the producer waits for every warp's x request
};

// CUDA-core decode of one (row group, unit) task: the lane's row (srow: the row at the unit's
// first byte) and half hf of every block's words; tot[m] += sum over its weights of w * x[m].
template <int TYPE>
__device__ __forceinline__ void fma_task(uint32_t srow, int hf, const float* xu, int K, int M, float (&tot)[kRsZs]) {
    using F = PnFmt<TYPE>;
    constexpr uint32_t MASK = (1u << F::BITS) - 1u;
    constexpr float BIAS = 12582912.0f + static_cast<float>(F::Z);  // 1.5 * 2^23 + z
    static_for<kUnitBlocks>([&](auto Bc) {
        constexpr int B = decltype(Bc)::value, OFF = kBlockBytes * B;
        const float d = (B & 1) ? half_hi(ld_shared_u32<OFF - 2>(srow)) : half_lo(ld_shared_u32<OFF>(srow));
        float blk[kRsZs] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int iw = 0; iw < 4; ++iw) {
            const int wi = 4 * hf + iw;
            const uint32_t wa = srow + static_cast<uint32_t>(OFF + 4 * wi);
            uint32_t wd;
            if constexpr (B & 1) {
                wd = ld_shared_u32<2>(wa);
            } else {
                wd = prmt(ld_shared_u32<0>(wa), ld_shared_u32<4>(wa), 0x5432u);  // bytes 2..5 of the pair
            }
            const float* xw = xu + B * F::BLK + F::CPW * wi;
#pragma unroll
            for (int t = 0; t < F::CPW; t += 2) {
                const int sh = F::BITS * (t >> 1);
                const float v0 = __uint_as_float(((wd >> sh) & MASK) | 0x4B400000u) - BIAS;
                const float v1 = __uint_as_float(((wd >> (sh + 16)) & MASK) | 0x4B400000u) - BIAS;
#pragma unroll
                for (int m = 0; m < kRsZs; ++m) {
                    if (m < M) {
                        const float2 xv = *reinterpret_cast<const float2*>(xw + static_cast<size_t>(m) * K + t);
                        blk[m] = fmaf(v1, xv.y, fmaf(v0, xv.x, blk[m]));
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kRsZs; ++m) tot[m] = fmaf(d, blk[m], tot[m]);
    });
}

template <int TYPE, int LR, bool SEG, bool FMA = false, int NT = 1>
__global__ void __launch_bounds__(kRsThreads, 1) pn_rows_kernel(const __grid_constant__ RsArgs a) {
    using C = Cfg<TYPE, NT, LR>;
    constexpr int ZS = rs_zs(NT);
    static_assert(!FMA || NT == 1, "the CUDA-core decode covers M <= 4");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t bar0 = smem_addr(base);
    const int S = a.S, M = a.M, nseg = SEG ? a.nseg : 1;
    const int CL = a.CL, cr = static_cast<int>(blockIdx.x) % CL, cid = static_cast<int>(blockIdx.x) / CL;
    const int ua = cr * a.U / CL, U = (cr + 1) * a.U / CL - ua;  // this CTA's K units [ua, ua + U)
    const int xk = U * C::UK;                                   // floats of an activation row it reads
    const int wpitch = rs_pitch(U * kUnitBytes);                // stage pitch of whole (CTA) rows
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t xfull = bar0 + 8u * (2 * S);      // all of x has landed (SEG)
    const uint32_t xreq = bar0 + 8u * (2 * S + 1);   // every consumer warp has requested its x
    const uint32_t xdone = bar0 + 8u * (2 * S + 2);  // every consumer warp has built its operands (x is dead)
    auto stage = [&](int s) { return base + a.off_stage + static_cast<uint32_t>(s) * a.stage_bytes; };
    auto rec = [&](int u) { return base + a.off_rec + static_cast<uint32_t>(u) * C::REC; };
    auto zbu = [&](int u) { return reinterpret_cast<float*>(base + a.off_zb) + u * rs_zb(NT); };
    __shared__ int seg_tab[kRsMaxSeg + 1];  // first unit of segment j (seg_tab[nseg] = U)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int active = SEG ? kRsWarps : min(kRsWarps, U);  // consumer warps with work
    const int64_t r0 = static_cast<int64_t>(cid) * a.N / a.G, r1 = static_cast<int64_t>(cid + 1) * a.N / a.G;
    const int nrows = static_cast<int>(r1 - r0);
    const int nstages = (nrows + kGroupRows - 1) / kGroupRows * nseg;  // (row group, segment), segment fastest
    float* part = reinterpret_cast<float*>(base + a.off_part);  // [warp][m][rows_pad]

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), kRsProducers);
            mbar_init(empty(s), active);
        }
        if (SEG) {
            for (int j = 0; j <= nseg; ++j) seg_tab[j] = j * U / nseg;
            mbar_init(xfull, 1);
        }
        mbar_init(xreq, active);
        mbar_init(xdone, active);
        mbar_fence_init();
    }
    __syncthreads();

    if (warp >= kRsWarps) {
        // ---------------- producers: one bulk copy per row, lane r of warp p copying row 8p + r ----------------
        const int pr = (warp - kRsWarps) * 8;  // the warp's first row of a group
        const uint64_t pol = l2_policy_evict_first();
        if (!(a.flags & kStaticWeights)) griddep_wait();  // W may be written by the previous grid
        bool ok = true;
        int s = 0;
        for (int i = 0, j = 0; s < nstages; ++s) {
            const int slot = s % S;
            if (s == a.x_ahead && !mbar_wait_warp(xreq, 0)) {
                ok = false;
                break;
            }
            if (s >= S && !mbar_wait_warp(empty(slot), ((s / S) - 1) & 1)) {
                ok = false;
                break;
            }
            if (s == a.x_slot0 && s < S && !mbar_wait_warp(xdone, 0)) {  // x lives in this slot until then
                ok = false;
                break;
            }
            // rows of the last group past the CTA's range are not copied: a row's products depend
            // on that row alone, and those rows' sums are never stored
            const int mine = min(8, max(0, nrows - i * kGroupRows - pr));
            int u0 = 0, bytes = U * kUnitBytes, pitch = wpitch;
            if (SEG) {
                u0 = seg_tab[j];
                bytes = (seg_tab[j + 1] - u0) * kUnitBytes;
                pitch = rs_pitch(bytes);
            }
            if (lane == 0) mbar_arrive_expect_tx(full(slot), static_cast<uint32_t>(mine * bytes));
            __syncwarp();
            if (lane < mine)
                bulk_g2s(smem_addr(stage(slot)) + static_cast<uint32_t>((pr + lane) * pitch),
                         a.W + (r0 + i * kGroupRows + pr + lane) * a.row_bytes + (ua + u0) * kUnitBytes,
                         static_cast<uint32_t>(bytes), full(slot), pol);
            if (++j == nseg) {
                j = 0;
                ++i;
            }
        }
        if (!ok && lane == 0) record_error(a.err, kErrEmptyWait);
        bool drained = true;  // every copy issued has landed before the CTA may exit
        for (int gg = max(0, s - S); drained && gg < s; ++gg) drained = mbar_wait_warp(full(gg % S), (gg / S) & 1);
        if (!drained && lane == 0) record_error(a.err, kErrDrainWait);
    } else if (warp < active) {
        // ---------------- consumer warps ----------------
        const int g = lane >> 2, c = lane & 3;
        const uint32_t sel = (c == 3) ? 0x7610u : 0x3210u;
        // the lane's B record and zero-point offsets per n8 tile (columns past 2M read a live
        // column's; their sums are never stored)
        uint32_t boff[NT];
        int mz[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            boff[t] = static_cast<uint32_t>((4 * min(g, max(0, 2 * M - 1 - 8 * t)) + c) * 16);
            mz[t] = min(4 * t + c, M - 1);
        }
        float* mine = part + warp * M * a.rows_pad;
        // one (row group, unit) task: rows g, g + 8 of the stage rows s0 / s8, at byte uo of them;
        // tot[t][h] += the row's sum for activation row 4t + c
        auto task = [&](uint32_t s0, uint32_t s8, uint32_t uo, int u, float (&tot)[NT][2]) {
            const uint32_t srow[2] = {s0 + uo, s8 + uo};
            const uint32_t srow_c[2] = {s0 + uo + 4u * c, s8 + uo + 4u * c};
            const uint32_t rs = smem_addr(rec(u));
            uint32_t srec[NT], srec_h[NT], szb[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                srec[t] = rs + boff[t];
                srec_h[t] = rs + boff[t] / 2;
                szb[t] = smem_addr(zbu(u)) + 4u * mz[t];
            }
            float acc[NT][2];
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.0f;
            pn_blocks<TYPE, NT, 0, 4, LR, ZS>(srow, srow_c, sel, srec, srec_h, szb, acc);
            pn_blocks<TYPE, NT, 4, 4, LR, ZS>(srow, srow_c, sel, srec, srec_h, szb, acc);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const float f = zbu(u)[kUnitBlocks * ZS + mz[t]];  // 2^(24 - sigma) of the unit
                tot[t][0] = fmaf(acc[t][0], f, tot[t][0]);
                tot[t][1] = fmaf(acc[t][1], f, tot[t][1]);
            }
        };
        // a task total of rows g, g + 8 of row group i into the warp's partials (+= in segments)
        auto store = [&](int i, const float (&tot)[NT][2], bool add) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (4 * t + c < M) {
                    float* pr = mine + (4 * t + c) * a.rows_pad + i * kGroupRows + g;
                    pr[0] = add ? pr[0] + tot[t][0] : tot[t][0];
                    pr[8] = add ? pr[8] + tot[t][1] : tot[t][1];
                }
        };
        bool ok = true;
        if constexpr (!SEG) {
            griddep_wait();  // X belongs to the previous grid until now
            // (unit, activation row) pairs of the warp's units, in order; x of pair q + 2 is in
            // flight while pair q builds
            float* xb = reinterpret_cast<float*>(base + a.off_x) + warp * 2 * C::UK;  // two x rows
            const int npair = ((U - warp + kRsWarps - 1) / kRsWarps) * M;
            auto load = [&](int q) {
                if (q < npair) {
                    const int u = warp + (q / M) * kRsWarps, m = q % M;
                    const float* src = a.X + static_cast<size_t>(m) * a.K + static_cast<size_t>(ua + u) * C::UK;
                    const uint32_t dst = smem_addr(xb + (q & 1) * C::UK);
                    for (int v = lane; v < C::UK / 4; v += 32) cp_async16(dst + 16u * v, src + 4 * v);
                }
                cp_async_commit();
            };
            load(0);
            load(1);
            __syncwarp();
            if (lane == 0) mbar_arrive(xreq);
            for (int q = 0; q < npair; ++q) {
                const int u = warp + (q / M) * kRsWarps, m = q % M;
                cp_async_wait<1>();  // pair q's x has landed (pair q + 1's may still be in flight)
                __syncwarp();
                build_row<TYPE, NT, LR, ZS>(rec(u), zbu(u), zbu(u) + kUnitBlocks * ZS, xb + (q & 1) * C::UK, m, lane);
                __syncwarp();
                load(q + 2);
            }
            cp_async_wait<0>();
            __syncwarp();
            if (lane == 0) mbar_arrive(xdone);
            for (int i = 0; i < nstages; ++i) {
                const int slot = i % S;
                if (!mbar_wait_warp(full(slot), (i / S) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t s0 = smem_addr(stage(slot)) + static_cast<uint32_t>(g * wpitch);
                const uint32_t s8 = s0 + static_cast<uint32_t>(8 * wpitch);
                float tot[NT][2];
#pragma unroll
                for (int t = 0; t < NT; ++t) tot[t][0] = tot[t][1] = 0.0f;
                for (int u = warp; u < U; u += kRsWarps) task(s0, s8, static_cast<uint32_t>(u * kUnitBytes), u, tot);
                store(i, tot, false);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(slot));
            }
        } else {
            for (int e = lane; e < M * a.rows_pad; e += 32) mine[e] = 0.0f;
            const float* xs = reinterpret_cast<const float*>(base + a.off_x);  // [M][xk]: the CTA's units of x
            if (warp == 0) {
                griddep_wait();  // X belongs to the previous grid until now
                if (lane == 0) {
                    const uint32_t row = static_cast<uint32_t>(xk) * 4u;
                    mbar_arrive_expect_tx(xfull, row * static_cast<uint32_t>(M));
                    for (int m = 0; m < M; ++m)
                        bulk_g2s_plain(smem_addr(xs) + m * row, a.X + static_cast<size_t>(m) * a.K + ua * C::UK, row,
                                       xfull);
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(xreq);
            ok = mbar_wait_warp(xfull, 0);
            if (ok && !FMA)
                for (int p = warp; p < U * M; p += kRsWarps) {
                    const int u = p / M, m = p - u * M;
                    build_row<TYPE, NT, LR, ZS>(rec(u), zbu(u), zbu(u) + kUnitBlocks * ZS,
                                                xs + static_cast<size_t>(m) * xk + u * C::UK, m, lane);
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(xdone);
            named_sync(kRsConsumerBar, 32 * kRsWarps);  // every unit's operands are built
            int k0 = warp;  // the warp's first task of the next stage (tasks of a stage: its units in order)
            for (int s = 0, i = 0, j = 0; ok && s < nstages; ++s) {
                const int slot = s % S;
                if (!mbar_wait_warp(full(slot), (s / S) & 1)) {
                    ok = false;
                    break;
                }
                const int u0 = seg_tab[j], n = seg_tab[j + 1] - u0;
                const uint32_t pitch = static_cast<uint32_t>(rs_pitch(n * kUnitBytes));
                const uint32_t s0 = smem_addr(stage(slot)) + g * pitch, s8 = s0 + 8u * pitch;
                if constexpr (FMA) {
                  if (k0 < n) {
                    float tot[kRsZs] = {0.0f, 0.0f, 0.0f, 0.0f};
                    const uint32_t srow = smem_addr(stage(slot)) + static_cast<uint32_t>(lane >> 1) * pitch;
                    for (int k = k0; k < n; k += kRsWarps)
                        fma_task<TYPE>(srow + static_cast<uint32_t>(k * kUnitBytes), lane & 1, xs + (u0 + k) * C::UK,
                                       xk, M, tot);
#pragma unroll
                    for (int m = 0; m < kRsZs; ++m) tot[m] += __shfl_xor_sync(0xffffffffu, tot[m], 1);
                    if ((lane & 1) == 0)
                        for (int m = 0; m < M; ++m) mine[m * a.rows_pad + i * kGroupRows + (lane >> 1)] += tot[m];
                  }
                } else if (k0 < n) {
                    float tot[NT][2];
#pragma unroll
                    for (int t = 0; t < NT; ++t) tot[t][0] = tot[t][1] = 0.0f;
                    for (int k = k0; k < n; k += kRsWarps) task(s0, s8, static_cast<uint32_t>(k * kUnitBytes), u0 + k, tot);
                    store(i, tot, true);
                }
                k0 = (k0 - n) & (kRsWarps - 1);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(slot));
                if (++j == nseg) {
                    j = 0;
                    ++i;
                }
            }
        }
        if (!ok && lane == 0) record_error(a.err, kErrFullWait);
    }

    // ---------------- the warps' row sums (and the cluster's, in CTA order) -> Y ----------------
    __syncthreads();
    if (CL == 1) {
        griddep_wait();  // Y may still be read by the previous grid
        for (int e = threadIdx.x; e < M * nrows; e += kRsThreads) {
            const int m = e / nrows, r = e - m * nrows;
            float v = 0.0f;
            for (int w = 0; w < active; ++w) v += part[(w * M + m) * a.rows_pad + r];
            a.Y[static_cast<size_t>(m) * a.N + r0 + r] = v;
        }
        return;
    }
    // this CTA's sum over its warps, in warp 0's slice; then CTA cr writes a share of the rows
    // from the sums of every CTA of the cluster (distributed shared memory)
    for (int e = threadIdx.x; e < M * nrows; e += kRsThreads) {
        const int m = e / nrows, r = e - m * nrows;
        float v = 0.0f;
        for (int w = 0; w < active; ++w) v += part[(w * M + m) * a.rows_pad + r];
        part[m * a.rows_pad + r] = v;
    }
    cluster_sync();
    griddep_wait();  // Y may still be read by the previous grid
    {
        const int E = M * nrows, e0 = cr * E / CL, e1 = (cr + 1) * E / CL;
        const uint32_t pbase = smem_addr(part);
        for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += kRsThreads) {
            const int m = e / nrows, r = e - m * nrows;
            const uint32_t off = 4u * static_cast<uint32_t>(m * a.rows_pad + r);
            float v = 0.0f;
            for (int q = 0; q < CL; ++q) v += ld_dsmem_f32(pbase + off, static_cast<uint32_t>(q));
            a.Y[static_cast<size_t>(m) * a.N + r0 + r] = v;
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its sums
}

struct RsPlan {
    int G = 0, CL = 1, S = 0, nseg = 0, rows_pad = 0, pitch = 0, x_slot0 = 0;
    uint32_t off_rec = 0, off_zb = 0, off_x = 0, off_part = 0, off_stage = 0, stage_bytes = 0, total = 0;
};

// Grid (clusters of CL CTAs, one CTA per SM, or one cluster per row when there are fewer rows),
// segments per row and the ring of stages, for the K units of one CTA (at most ceil(U / CL)).
// Rows of at most 16 units stay whole (per-warp x buffers); longer rows are cut into segments of
// at most 8, 6 then 4 units (all of the CTA's x staged). x is read only while the operands are
// built, so it may sit in the ring's last slots (slot 2 or later), which the producer fills only
// once every warp has built: of the two layouts, x apart or x in the ring, the one with the deeper
// ring is taken (8..3 stages, then 2 as a last resort). The CUDA-core decode (fma) keeps no B
// operands and reads x throughout, so its x has a region of its own. False when nothing fits.
template <int TYPE, int LR, int NT = 1>
bool rs_plan(int64_t N, int Ut, int M, int sms, int s_req, RsPlan& p, bool fma = false, bool x_in_ring = true,
             int CL = 1, int max_clusters = 0) {
    using C = Cfg<TYPE, NT, LR>;
    if (CL < 1 || CL > 8 || sms / CL < 1 || Ut < CL || (fma && NT > 1)) return false;
    const int U = (Ut + CL - 1) / CL;  // the most units of a CTA
    if (U < 1 || M < 1 || M > rs_zs(NT) || (U + 3) / 4 > kRsMaxSeg) return false;
    p.CL = CL;
    // clusters: one CTA per SM, no more than can be resident at once (max_clusters > 0)
    const int ncl = max_clusters > 0 ? std::min(sms / CL, max_clusters) : sms / CL;
    p.G = static_cast<int>(std::min<int64_t>(ncl, N));
    const int64_t rows_max = (N + p.G - 1) / p.G;
    p.rows_pad = static_cast<int>((rows_max + kGroupRows - 1) / kGroupRows * kGroupRows);
    const bool whole = U <= kRsWholeUnits;
    const uint32_t nrec = fma ? 0u : static_cast<uint32_t>(U);
    p.off_rec = align_up(8u * (2u * kMaxStages + 3), 128);
    p.off_zb = align_up(p.off_rec + nrec * C::REC, 16);
    p.off_part = align_up(p.off_zb + nrec * rs_zb(NT) * 4u, 16);
    const uint32_t part_end = p.off_part + kRsWarps * static_cast<uint32_t>(M * p.rows_pad) * 4u;
    const uint32_t xbytes =
        (whole && !fma) ? kRsWarps * 2u * C::UK * 4u : static_cast<uint32_t>(M) * U * C::UK * 4u;
    const uint32_t sep_x = align_up(part_end, 16), sep_stage = align_up(sep_x + xbytes, 128);
    const uint32_t ovl_stage = align_up(part_end, 128);
    const int cap[3] = {8, 6, 4};
    const int s_hi = s_req > 0 ? s_req : 8;
    for (int s_lo : {3, 2})
        for (int t = 0; t < (whole ? 1 : 3); ++t) {
            p.nseg = whole ? 1 : (U + cap[t] - 1) / cap[t];
            const int longest = (U + p.nseg - 1) / p.nseg;
            p.pitch = rs_pitch(longest * kUnitBytes);
            p.stage_bytes = align_up(static_cast<uint32_t>(kGroupRows * p.pitch), 128);
            const int nx = static_cast<int>((xbytes + p.stage_bytes - 1) / p.stage_bytes);
            const int lo = s_req > 0 ? s_req : s_lo;
            int s_sep = 0, s_ovl = 0;
            for (int S = std::min(s_hi, kMaxStages); S >= lo && s_sep == 0; --S)
                if (sep_stage + static_cast<uint32_t>(S) * p.stage_bytes + 1024u <= kSmemOne) s_sep = S;
            for (int S = std::min(s_hi, kMaxStages); S >= lo && s_ovl == 0 && !fma && x_in_ring; --S)
                if (S - nx >= 2 && ovl_stage + static_cast<uint32_t>(S) * p.stage_bytes + 1024u <= kSmemOne) s_ovl = S;
            if (s_sep == 0 && s_ovl == 0) continue;
            const bool ovl = s_ovl > s_sep;
            p.S = ovl ? s_ovl : s_sep;
            p.off_stage = ovl ? ovl_stage : sep_stage;
            p.x_slot0 = ovl ? p.S - nx : p.S;
            p.off_x = ovl ? p.off_stage + static_cast<uint32_t>(p.x_slot0) * p.stage_bytes : sep_x;
            p.total = p.off_stage + static_cast<uint32_t>(p.S) * p.stage_bytes;
            return true;
        }
    return false;
}

template <int TYPE, int LR, bool SEG, bool FMA = false, int NT = 1>
cudaError_t launch_rows_kernel(const RsArgs& a, const RsPlan& p, cudaStream_t stream) {
    auto kern = pn_rows_kernel<TYPE, LR, SEG, FMA, NT>;
    static std::atomic<bool> opted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!opted[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemOne));
        if (e != cudaSuccess) return e;
        opted[dev].store(true, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(p.G * p.CL, 1, 1);
    lc.blockDim = dim3(kRsThreads, 1, 1);
    lc.dynamicSmemBytes = p.total + 1024u;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.CL);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, kern, a);
}

// Estimated time (us) of a row-stream plan, fitted to the decode-step projections on this GPU at
// M = 1, 2, 4 with every cluster size forced: ~2.5 us until the first stage is multiplied; 0.35 us
// per further (unit, activation row) operand build of the busiest warp (whole rows: warp w builds
// units w, w + 8, ..; segments: the builds are dealt evenly); then the longer of the busiest
// consumer warp's tasks (0.65 us per 16 rows x one unit) and the CTA's weight stream (35 GB/s per
// SM, and at least ~0.8 us per stage of 16 copies however small they are); plus 1.5 us for a
// cluster's final sum and 4 us for segments (all builds before any task).
inline double rs_cost(const RsPlan& p, int64_t N, int Ut, int M, int NT = 1) {
    const int U = (Ut + p.CL - 1) / p.CL;
    const int64_t rows = (N + p.G - 1) / p.G;
    const int64_t groups = (rows + kGroupRows - 1) / kGroupRows;
    const bool seg = p.nseg > 1;
    const int per_warp = (U + kRsWarps - 1) / kRsWarps;
    const double tasks = seg ? static_cast<double>((groups * U + kRsWarps - 1) / kRsWarps)
                             : static_cast<double>(groups * per_warp);
    const double builds = seg ? static_cast<double>((U * M + kRsWarps - 1) / kRsWarps) : static_cast<double>(per_warp * M);
    const double stream = std::max(static_cast<double>(rows) * U * kUnitBytes / 35e3, 0.8 * static_cast<double>(groups * p.nseg));
    const double per_task = NT == 1 ? 0.65 : 0.65 * 1.4;  // a second n8 tile shares the decode
    return 2.5 + 0.35 * (builds - 1.0) + std::max(per_task * tasks, stream) + (p.CL > 1 ? 1.5 : 0.0) +
           (seg ? 4.0 : 0.0);
}

// The cheapest plan over clusters of 1, 2, 4 and 8 CTAs (cl_req > 0: that size only).
// resident(CL, plan) = clusters of CL CTAs of that plan's kernel that fit on the GPU at once
// (clusters of 4 or 8 need that many SMs of one GPC, which does not divide every GPC).
template <int TYPE, int LR, int NT, class Resident>
bool rs_best_plan(int64_t N, int U, int M, int sms, int s_req, bool fma, bool x_in_ring, int cl_req, RsPlan& p,
                  Resident&& resident) {
    bool found = false;
    double best = 0.0;
    for (int CL : {1, 2, 4, 8}) {
        if (cl_req > 0 && CL != cl_req) continue;
        RsPlan q;
        if (!rs_plan<TYPE, LR, NT>(N, U, M, sms, s_req, q, fma, x_in_ring, CL)) continue;
        if (CL > 1) {
            const int most = resident(CL, q);
            if (most < 1) continue;
            if (most < q.G && !rs_plan<TYPE, LR, NT>(N, U, M, sms, s_req, q, fma, x_in_ring, CL, most)) continue;
        }
        const double cost = rs_cost(q, N, U, M, NT);
        if (!found || cost < best) {
            p = q;
            best = cost;
            found = true;
        }
    }
    return found;
}

// Clusters of CL CTAs of the plan's kernel that can be resident at once on this device (0 when the
// query fails).
template <int TYPE, int LR, int NT>
int rows_resident_clusters(int CL, const RsPlan& q, bool fma) {
    void (*kern)(RsArgs) = (fma && NT == 1) ? pn_rows_kernel<TYPE, LR, true, NT == 1, NT>
                           : (q.nseg > 1 ? pn_rows_kernel<TYPE, LR, true, false, NT> : pn_rows_kernel<TYPE, LR, false, false, NT>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemOne)) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(q.G * CL, 1, 1);
    lc.blockDim = dim3(kRsThreads, 1, 1);
    lc.dynamicSmemBytes = q.total + 1024u;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// rs_best_plan with the device's SM count and resident clusters, cached per device and shape.
template <int TYPE, int LR, int NT>
bool rs_cached_plan(int64_t N, int U, int M, int s_req, bool fma, bool x_in_ring, int cl_req, RsPlan& p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    using Key = std::tuple<int, int64_t, int, int, int, bool, bool, int>;
    static std::mutex mu;
    static std::map<Key, RsPlan> cache;
    const Key key{dev, N, U, M, s_req, fma, x_in_ring, cl_req};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            p = it->second;
            return true;
        }
    }
    auto resident = [fma](int CL, const RsPlan& q) { return rows_resident_clusters<TYPE, LR, NT>(CL, q, fma); };
    if (!rs_best_plan<TYPE, LR, NT>(N, U, M, device_sm_count(), s_req, fma, x_in_ring, cl_req, p, resident)) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.emplace(key, p);
    return true;
}

template <int TYPE, int LR, int NT = 1>
cudaError_t launch_rows(const uint8_t* W, const float* X, float* Y, int* err, int64_t N, int64_t K, int M, int U,
                        int row_bytes, int s_req, bool static_weights, bool fma, int x_ahead, bool x_in_ring,
                        int cl_req, cudaStream_t stream) {
    RsPlan p;
    if ((fma && NT > 1) || !rs_cached_plan<TYPE, LR, NT>(N, U, M, s_req, fma, x_in_ring, cl_req, p))
        return cudaErrorNotSupported;
    RsArgs a{};
    a.W = W;
    a.X = X;
    a.Y = Y;
    a.err = err;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.U = U;
    a.G = p.G;
    a.CL = p.CL;
    a.S = p.S;
    a.nseg = p.nseg;
    a.row_bytes = row_bytes;
    a.pitch = p.pitch;
    a.rows_pad = p.rows_pad;
    a.flags = static_weights ? kStaticWeights : 0u;
    a.off_rec = p.off_rec;
    a.off_zb = p.off_zb;
    a.off_x = p.off_x;
    a.off_part = p.off_part;
    a.off_stage = p.off_stage;
    a.stage_bytes = p.stage_bytes;
    a.x_slot0 = p.x_slot0;
    a.x_ahead = x_ahead;
    if constexpr (NT == 1)
        if (fma) return launch_rows_kernel<TYPE, LR, true, true>(a, p, stream);
    return p.nseg > 1 ? launch_rows_kernel<TYPE, LR, true, false, NT>(a, p, stream)
                      : launch_rows_kernel<TYPE, LR, false, false, NT>(a, p, stream);
}

template <int TYPE>
cudaError_t launch_rows_typed(const uint8_t* W, const float* X, float* Y, int* err, int64_t N, int64_t K, int M,
                              int U, int row_bytes, int s_req, bool static_weights, bool fma, int xa, bool xr,
                              int cl, cudaStream_t stream) {
    switch (M) {
        case 1: return launch_rows<TYPE, 8>(W, X, Y, err, N, K, M, U, row_bytes, s_req, static_weights, fma, xa, xr, cl, stream);
        case 2: return launch_rows<TYPE, 16>(W, X, Y, err, N, K, M, U, row_bytes, s_req, static_weights, fma, xa, xr, cl, stream);
        case 3: return launch_rows<TYPE, 24>(W, X, Y, err, N, K, M, U, row_bytes, s_req, static_weights, fma, xa, xr, cl, stream);
        case 4: return launch_rows<TYPE, 32>(W, X, Y, err, N, K, M, U, row_bytes, s_req, static_weights, fma, xa, xr, cl, stream);
        case 5:
        case 6:
        case 7:
        case 8:
            return launch_rows<TYPE, 32, 2>(W, X, Y, err, N, K, M, U, row_bytes, s_req, static_weights, fma, xa, xr, cl,
                                            stream);
        default: return cudaErrorNotSupported;
    }
}

template <class F>
cudaError_t launch_policy(const CUtensorMap (&map)[2], const float* X, float* Y, int* err, int64_t N, int64_t K,
                          int M, int U, const int (&req)[3], bool static_weights, cudaStream_t stream) {
    KArgs<F> ka{};
    ka.map[0] = map[0];
    ka.map[1] = map[1];
    ka.c.X = X;
    ka.c.Y = Y;
    ka.c.err = err;
    ka.c.N = static_cast<int>(N);
    ka.c.K = static_cast<int>(K);
    ka.c.M = M;
    return cl_launch<F>(ka, N, U, req, static_weights, stream);
}

template <int TYPE>
cudaError_t launch_typed(const CUtensorMap (&map)[2], const float* X, float* Y, int* err, int64_t N, int64_t K, int M,
                         int U, const int (&req)[3], bool static_weights, cudaStream_t stream) {
    const int nt = (2 * M + 7) / 8;
    if (nt == 1) return launch_policy<PnMma<TYPE, 1>>(map, X, Y, err, N, K, M, U, req, static_weights, stream);
    if (nt == 2) return launch_policy<PnMma<TYPE, 2>>(map, X, Y, err, N, K, M, U, req, static_weights, stream);
    return launch_policy<PnMma<TYPE, 4>>(map, X, Y, err, N, K, M, U, req, static_weights, stream);
}

}  // namespace

cudaError_t launch_pn_gemv_mma(int type, const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y,
                               int* err, int c_req, int s_req, bool static_weights, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int blk = (type == kTypePn3t) ? 80 : 64;
    const int64_t nb = K / blk;
    if (nb % kUnitBlocks != 0 || M < 1 || M > 16) return cudaErrorNotSupported;
    const int64_t U = nb / kUnitBlocks;
    if (N > INT32_MAX - 64 || K > INT32_MAX || U * kUnitU32 > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || reinterpret_cast<uintptr_t>(X) % 16 != 0)
        return cudaErrorNotSupported;
    CUtensorMap map[2];
    if (!encode_u32_map(&map[0], W, N, nb * kBlockBytes / 4, kUnitU32, kPieceRows) ||
        !encode_u32_map(&map[1], W, N, nb * kBlockBytes / 4, kUnitU32, kStageRows))
        return cudaErrorNotSupported;
    // PNQ_PN_CFG = "CTAs per cluster, stages, CTAs per SM, path (1 rows, 2 strips), decode (1 CUDA-core FMA),
    // row stream: weight stages issued before x is requested (0: 1), x apart from the ring (1), CTAs per
    // cluster splitting K (1, 2, 4, 8; 0: cheapest)"
    static int env[8];
    static std::once_flag once;
    std::call_once(once, [] { env_cluster_config("PNQ_PN_CFG", env); });
    const int req[3] = {c_req > 0 ? c_req : env[0], s_req > 0 ? s_req : env[1], env[2]};
    // the row stream (M <= 8) when its plan fits, else the strip pipeline
    const int row_bytes = static_cast<int>(nb * kBlockBytes);
    const bool fma = env[4] == 1;
    const int x_ahead = env[5] > 0 ? env[5] : 1;
    const bool x_in_ring = env[6] != 1;
    const int rows_cl = env[7];
    if (env[3] != 2 && M <= 8 && c_req <= 0) {
        const cudaError_t e = (type == kTypePn3t)
                                  ? launch_rows_typed<kTypePn3t>(W, X, Y, err, N, K, M, static_cast<int>(U), row_bytes,
                                                                 req[1], static_weights, fma, x_ahead, x_in_ring, rows_cl, stream)
                                  : launch_rows_typed<kTypePn4t>(W, X, Y, err, N, K, M, static_cast<int>(U), row_bytes,
                                                                 req[1], static_weights, fma, x_ahead, x_in_ring, rows_cl, stream);
        if (e != cudaErrorNotSupported || env[3] == 1 || fma) return e;
    }
    return (type == kTypePn3t)
               ? launch_typed<kTypePn3t>(map, X, Y, err, N, K, M, static_cast<int>(U), req, static_weights, stream)
               : launch_typed<kTypePn4t>(map, X, Y, err, N, K, M, static_cast<int>(U), req, static_weights, stream);
}

}  // namespace pnq
