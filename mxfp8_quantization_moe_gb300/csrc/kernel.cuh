// kernel.cuh -- the persistent tile kernel shared by every entry point.
//
// One CTA per SM (or a few): (TM/32)*4 consumer warps and one producer warp.
// The producer's lane 0 streams the input tiles (TM rows x 128 bf16 columns
// per tensor, as two 64-column boxes with the 128-byte swizzle) into a ring
// of shared-memory stages with TMA; each stage has a "full" mbarrier
// (transaction bytes) and an "empty" mbarrier (one arrive per consumer warp).
//
// Consumer warp w owns the 32 x 32 sub-tile (row block w/4, column block w%4)
// of every tile, so no two warps ever share data and the only
// synchronisation inside a tile is __syncwarp.  Lane l owns one whole
// 32-element block at a time, so a block's amax, scale and codes need no
// cross-lane traffic:
//   row pass: lane l takes sub-tile row l (four 16-byte chunks per input),
//             runs the element op, encodes the 1x32 block and stores its 32
//             codes (32 contiguous bytes of the row-major output);
//   col pass: the warp transposes its sub-tile in place (ldmatrix.trans of
//             four 32x8 column units, stmatrix of the rows they become), and
//             lane l then treats row l of the transposed sub-tile -- column l
//             of the original -- exactly like the row pass, storing 32
//             contiguous bytes of the column-major output.
// In "both" mode the row pass writes the bf16 element values back into the
// stage (over an input it no longer needs), so both scale sets come from one
// read of the inputs; "col" mode transposes the inputs and runs the element
// op on the transposed rows.
//
// Every wait is bounded (about a second); on time-out the kernel sets a bit in
// the status word and returns, after the producer has waited (bounded) for
// the loads it issued.
#pragma once

#include "device.cuh"

namespace mx {

template <int OP>
struct OpTraits;
template <>
struct OpTraits<kQuant> {
    static constexpr int kIn = 1, kOut = 1;
};
template <>
struct OpTraits<kFwd> {
    static constexpr int kIn = 2, kOut = 1;
};
template <>
struct OpTraits<kBwd> {
    static constexpr int kIn = 3, kOut = 2;
};

// Tile height, pipeline depth, resident CTAs per SM and row-scale group
// (consecutive column tiles a CTA takes in a row, so that their row scales
// leave as one 4*GROUP-byte store per row; it pays in the "both" modes, the
// plain tile-cyclic order is faster elsewhere) for each instantiation: more warps hide more latency where registers and shared
// memory allow it (the cast alone needs few registers).  Registers are
// granted per four warps, so the producer warp costs three warps' worth: 17
// warps get at most 96 registers a thread, 13 warps 128.
template <int OP, int MODE>
struct Tuning;
#define MX_TUNE(OP, MODE, TM, STAGES, CTAS, GROUP)                                   \
    template <>                                                                      \
    struct Tuning<OP, MODE> {                                                        \
        static constexpr int kTM = TM, kStages = STAGES, kCtas = CTAS, kGroup = GROUP; \
        static_assert((TM / 32) * 4 + 1 <= 32, "at most 1024 threads per CTA");     \
    };
MX_TUNE(kQuant, kRow, 192, 3, 1, 1)
MX_TUNE(kQuant, kCol, 192, 3, 1, 1)
MX_TUNE(kQuant, kBoth, 192, 3, 1, 4)
MX_TUNE(kFwd, kRow, 128, 3, 1, 1)
MX_TUNE(kFwd, kCol, 128, 3, 1, 1)
MX_TUNE(kFwd, kBoth, 128, 3, 1, 4)
MX_TUNE(kBwd, kRow, 96, 3, 1, 1)
MX_TUNE(kBwd, kCol, 96, 3, 1, 1)
MX_TUNE(kBwd, kBoth, 128, 2, 1, 2)
#undef MX_TUNE

// The same per activation and scale kind: GEGLU's backward "both" with
// plain scales takes 96-row tiles with three stages and keeps its values in
// registers (its policy then is the rational tail, the tail table having no
// room there): 2223 -> 2160 us at 131072 x 8192, where SwiGLU's measured no
// gain from that shape, and the per-group one lost 12 % (2282 -> 2551).
template <int OP, int MODE, int ACT, bool GRP>
struct TuningFor : Tuning<OP, MODE> {
};
template <>
struct TuningFor<kBwd, kBoth, kGelu, false> {
    static constexpr int kTM = 96, kStages = 3, kCtas = 1, kGroup = 2;
};

// The activation policy a kernel evaluates: GEGLU's tail table for the
// forward and the per-group backward "both" (two stages of 128-row tiles),
// its rational tail for the rest of the backward (three stages of 96-row
// tiles leave no room for the table; two stages measured 11-14 % slower in
// the row and column modes, and the table with two stages of 128 rows 3 %
// slower in "both").
template <int OP, int MODE, int ACT, bool GRP>
constexpr int policy_of()
{
    return (ACT == kGelu && OP == kBwd && (MODE != kBoth || !GRP)) ? kGeluPoly : ACT;
}

// static shared memory of the policy's kernels: the tail table (Phi by sign
// for the forward, (L, Q) pairs for the backward)
template <int OP, int POL>
constexpr size_t static_smem_bytes()
{
    return POL != kGelu ? 0 : sizeof(float2) * kGeluTabN;
}

template <int TM>
__host__ __device__ constexpr int warps_of() { return (TM / kSub) * (kTileN / kSub); }

template <int TM>
__host__ __device__ constexpr int tile_bytes() { return TM * kTileN * 2; }

// row-scale bytes of one group of G column tiles and one output: 4 G per row
// (one per 32-column block)
template <int TM, int G>
__host__ __device__ constexpr int scale_group_bytes() { return TM * 4 * G; }

// shared memory: 1 KB alignment slack, the stages, the row-scale buffers
// (a ring of STAGES + 1 groups, per output), the mbarriers
template <int OP, int TM, int STAGES, int G, bool GRP>
constexpr size_t smem_bytes()
{
    return 1024 + static_cast<size_t>(STAGES) * OpTraits<OP>::kIn * tile_bytes<TM>() +
           static_cast<size_t>(STAGES + 1) * OpTraits<OP>::kOut * scale_group_bytes<TM, G>() + 4 * STAGES * 8 +
           (GRP ? kGroupTableBytes : 0);
}

// ------------------------------------------------------------ block values
// Bit p: pair p of chunk c (in the slot, 16-byte offset roff_c) has a fast
// value near a rounding midpoint -- the block_values test again, for the
// rare blocks where some value is.
template <int OP, int ACT>
static __device__ __noinline__ uint32_t near_bits_chunk(const uint8_t *stage, int tile_bytes_, uint32_t roff_c)
{
    constexpr int NIN = OpTraits<OP>::kIn;
    uint32_t in[3][4];
#pragma unroll
    for (int k = 0; k < NIN; ++k) {
        const uint4 v = *reinterpret_cast<const uint4 *>(stage + k * tile_bytes_ + roff_c);
        in[k][0] = v.x;
        in[k][1] = v.y;
        in[k][2] = v.z;
        in[k][3] = v.w;
    }
    uint32_t near = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if constexpr (OP == kFwd) {
            near |= static_cast<uint32_t>(near_mid2(Gated<ACT>::h2(in[0][p], in[1][p]), Gated<ACT>::kWinH)) << p;
        } else {
            uint64_t DG, DU;
            Gated<ACT>::grads2(in[0][p], in[1][p], in[2][p], DG, DU);
            near |= static_cast<uint32_t>(near_mid2(DG, Gated<ACT>::kWinDgate) | near_mid2(DU, Gated<ACT>::kWinDup)) << p;
        }
    }
    return near;
}

// The rare path of one pair of elements, out of line (scalar arguments and a
// 64-bit result, so that calling it costs the common path nothing): the
// pair's fast values evaluated again, then, element by element, the exact
// (correctly rounded) value where the block is recomputed whole (`whole`: a
// huge or infinite value), where the gate lies outside the fast range (the
// exact path settles gates below it on its wide-range route), where a fast
// value is not finite or where it lies near a 0x60/0x61 rounding midpoint;
// the fast value elsewhere.
// w0, w1, w2: the pair's input words in the op's order (gate, up or dh,
// gate, up); ta, tb: the activation's exact-path tables.  Returns the output
// words (the second output's in the high half).
template <int OP, int ACT>
static __device__ __noinline__ uint64_t settle_pair(const void *ta, const void *tb, uint32_t w0, uint32_t w1,
                                                    uint32_t w2, bool whole)
{
    constexpr int kGate = OP == kFwd ? 0 : 1;
    const uint32_t gw = kGate == 0 ? w0 : w1;
    uint64_t V0, V1 = 0;
    if constexpr (OP == kFwd)
        V0 = Gated<ACT>::h2(w0, w1);
    else
        Gated<ACT>::grads2(w0, w1, w2, V0, V1);
    float v0[2] = {f2lo(V0), f2hi(V0)}, v1[2] = {f2lo(V1), f2hi(V1)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t gb = h ? gw >> 16 : gw & 0xFFFFu;
        bool need = whole || far_gate<ACT>(gb) || !isfinite(v0[h]);
        if constexpr (OP == kFwd)
            need |= near_mid1(v0[h], Gated<ACT>::kWinH);
        else
            need |= !isfinite(v1[h]) || near_mid1(v0[h], Gated<ACT>::kWinDgate) || near_mid1(v1[h], Gated<ACT>::kWinDup);
        if (need) {
            const float x0 = h ? bf16hi(w0) : bf16lo(w0), x1 = h ? bf16hi(w1) : bf16lo(w1);
            if constexpr (OP == kFwd) {
                v0[h] = Gated<ACT>::h_exact(ta, tb, x0, x1);
            } else {
                const float2 r = Gated<ACT>::grads_exact(ta, tb, x0, x1, h ? bf16hi(w2) : bf16lo(w2));
                v0[h] = r.x;
                v1[h] = r.y;
            }
        }
    }
    return static_cast<uint64_t>(pack_bf16x2(v0[0], v0[1])) | (static_cast<uint64_t>(pack_bf16x2(v1[0], v1[1])) << 32);
}

// word p (0..3) of the 16-byte chunk at roff_c of the slot at `slot_base`
__device__ __forceinline__ uint32_t word_at(const uint8_t *slot_base, uint32_t roff_c, int p)
{
    return *reinterpret_cast<const uint32_t *>(slot_base + roff_c + 4 * p);
}

// settle_pair on every flagged pair of the warp (bit j of `near`: pair j of
// the lane's block, whose chunk j / 4 sits at r0..r3 in the slots), for
// blocks whose flagged pairs span more than two pair numbers in the warp
// (a row of far gates, whose lane owns all 16 pairs, in a row pass): the
// warp's flagged pairs are numbered across the lanes and lane t of a round
// takes pair base + t (its owner found by a search over the owners' first
// numbers), so such a block costs about one settle_pair per round rather
// than one per pair in turn.  Each result is left in the stage over the
// pair's words of slot 0 (and of slot 1 for the second output), for the
// lanes to read back.  Out of line, with scalar arguments, so that none of
// this weighs on the callers' registers.  Used by the forward's row passes
// (mixed 4096 x 7168: row 102 -> 47 us, col 104 -> 49, both 119 -> 61); the
// backward's row pass gained as much on that workload but lost 1.8 % on the
// large one (code placement).
template <int OP, int ACT>
static __device__ __noinline__ void settle_flagged(const void *ta, const void *tb, uint8_t *stage, int tile_bytes_,
                                                   uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t near,
                                                   bool whole)
{
    constexpr int NIN = OpTraits<OP>::kIn;
    constexpr int NOUT = OpTraits<OP>::kOut;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t cnt = __popc(near);
    uint32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= static_cast<uint32_t>(d)) incl += v;
    }
    const uint32_t excl = incl - cnt;
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    for (uint32_t base = 0; base < total; base += 32) {
        const uint32_t k = base + lane;
        int owner = 0;            // the last lane whose first number is <= k
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
            const uint32_t e = __shfl_sync(0xFFFFFFFFu, excl, owner + step);
            if (e <= k) owner += step;
        }
        const uint32_t nm = __shfl_sync(0xFFFFFFFFu, near, owner);
        const uint32_t first = __shfl_sync(0xFFFFFFFFu, excl, owner);
        const bool wh = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(whole), owner) != 0u;
        const uint32_t o0 = __shfl_sync(0xFFFFFFFFu, r0, owner), o1 = __shfl_sync(0xFFFFFFFFu, r1, owner);
        const uint32_t o2 = __shfl_sync(0xFFFFFFFFu, r2, owner), o3 = __shfl_sync(0xFFFFFFFFu, r3, owner);
        if (k < total) {
            const int j = static_cast<int>(__fns(nm, 0u, static_cast<int>(k - first) + 1));
            const int p = j & 3;
            const uint32_t rc = (j >> 2) == 0 ? o0 : (j >> 2) == 1 ? o1 : (j >> 2) == 2 ? o2 : o3;
            const uint64_t r = settle_pair<OP, ACT>(ta, tb, word_at(stage, rc, p), word_at(stage + tile_bytes_, rc, p),
                                                    NIN > 2 ? word_at(stage + 2 * tile_bytes_, rc, p) : 0u, wh);
            *reinterpret_cast<uint32_t *>(stage + rc + 4 * p) = static_cast<uint32_t>(r);
            if constexpr (NOUT > 1)
                *reinterpret_cast<uint32_t *>(stage + tile_bytes_ + rc + 4 * p) = static_cast<uint32_t>(r >> 32);
        }
    }
    __syncwarp();
}

// Element values of the lane's block.  For the cast, the input itself; for
// the gated ops, the fast element op on the NIN input slots and the midpoint
// test of every value (near_mid2: a value within its window of a 0x60/0x61
// rounding midpoint, where a scale byte could step); then, for the warps with
// a lane whose block holds a flagged value, a gate outside the fast range or
// a huge, infinite or NaN amax, settle_pair on the flagged pairs (on every
// pair of a chunk holding such a gate, of a block with such an amax): lane
// by lane, or (COOP, the forward's row passes) across the warp's lanes
// where the flagged pairs span more than two pair numbers (settle_flagged).
// (Testing every value, rather than
// only the blocks whose amax sits at that mantissa pair, also covers the
// other direction's blocks in "both" mode, and measured cheaper than scanning
// the risky blocks.)  DIST (forward only): the test keeps a running minimum
// of the values' distances instead of a bit per pair, and the flagged pairs
// are found again in the rare path.  Returns the outputs' amax patterns.
template <int OP, int ACT, bool DIST = false, bool COOP = OP == kFwd>
__device__ __forceinline__ void block_values(const KernelArgs &a, const uint8_t *stage, int tile_bytes_,
                                             const uint32_t (&roff)[4], uint32_t (&out)[2][16],
                                             uint32_t (&amax)[2])
{
    constexpr int NOUT = OpTraits<OP>::kOut;
    constexpr int NIN = OpTraits<OP>::kIn;
    uint32_t dmin = 0xFFFFFFFFu;
    uint32_t near = 0;     // bit j: pair j (elements 2j, 2j+1)
    uint32_t farc = 0;     // bit c: chunk c holds a gate outside the fast range
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t in[3][4];
#pragma unroll
        for (int k = 0; k < NIN; ++k) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + k * tile_bytes_ + roff[c]);
            in[k][0] = v.x;
            in[k][1] = v.y;
            in[k][2] = v.z;
            in[k][3] = v.w;
        }
        if constexpr (OP == kQuant) {
#pragma unroll
            for (int p = 0; p < 4; ++p) out[0][4 * c + p] = in[0][p];
        } else if constexpr (OP == kFwd) {
            farc |= gates_fast8(in[0], Gated<ACT>::kMinGate2) ? 0u : 1u << c;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint64_t H = Gated<ACT>::h2(in[0][p], in[1][p]);
                out[0][4 * c + p] = pack_bf16x2(f2lo(H), f2hi(H));
                if constexpr (DIST)
                    dmin = min(dmin, mid_dist2(H, Gated<ACT>::kWinH));
                else
                    near |= static_cast<uint32_t>(near_mid2(H, Gated<ACT>::kWinH)) << (4 * c + p);
            }
        } else {
            farc |= gates_fast8(in[1], Gated<ACT>::kMinGate2) ? 0u : 1u << c;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint64_t DG, DU;
                Gated<ACT>::grads2(in[0][p], in[1][p], in[2][p], DG, DU);
                out[0][4 * c + p] = pack_bf16x2(f2lo(DG), f2hi(DG));
                out[1][4 * c + p] = pack_bf16x2(f2lo(DU), f2hi(DU));
                near |= static_cast<uint32_t>(near_mid2(DG, Gated<ACT>::kWinDgate) | near_mid2(DU, Gated<ACT>::kWinDup)) << (4 * c + p);
            }
        }
    }
#pragma unroll
    for (int o = 0; o < NOUT; ++o) amax[o] = amax32_lane(out[o]);
    if constexpr (OP != kQuant) {
        bool full = false, nanb = false;
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
            full |= huge_amax(amax[o]);
            nanb |= nan_amax(amax[o]);
        }
        if (__any_sync(0xFFFFFFFFu, near != 0u || dmin == 0u || full || nanb || farc != 0u)) {
            if constexpr (DIST && OP == kFwd) {
                // which pairs: those near a midpoint (their fast values
                // evaluated again), unless every pair is settled anyway
                if (!full && dmin == 0u) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) near |= near_bits_chunk<OP, ACT>(stage, tile_bytes_, roff[c]) << (4 * c);
                }
            }
            // every pair of a chunk holding a gate outside the fast range, of
            // the whole block if a value is huge or infinite
#pragma unroll
            for (int c = 0; c < 4; ++c) near |= ((farc >> c) & 1u) ? 0xFu << (4 * c) : 0u;
            if (full || nanb) near = 0xFFFFu;
            bool coop = false;
            if constexpr (COOP) coop = __popc(__reduce_or_sync(0xFFFFFFFFu, near)) > 2;
            if (coop) {
                settle_flagged<OP, ACT>(Gated<ACT>::table_a(a), Gated<ACT>::table_b(a), const_cast<uint8_t *>(stage),
                                        tile_bytes_, roff[0], roff[1], roff[2], roff[3], near, full);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if ((near >> j) & 1u) {
                        out[0][j] = word_at(stage, roff[j >> 2], j & 3);
                        if constexpr (NOUT > 1) out[1][j] = word_at(stage + tile_bytes_, roff[j >> 2], j & 3);
                    }
                }
            } else {
                // few pair numbers flagged: each lane settles its own
                const void *ta = Gated<ACT>::table_a(a), *tb = Gated<ACT>::table_b(a);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if ((near >> j) & 1u) {
                        const uint32_t cj = roff[j >> 2];
                        const uint64_t r = settle_pair<OP, ACT>(ta, tb, word_at(stage, cj, j & 3),
                                                                word_at(stage + tile_bytes_, cj, j & 3),
                                                                NIN > 2 ? word_at(stage + 2 * tile_bytes_, cj, j & 3) : 0u,
                                                                full);
                        out[0][j] = static_cast<uint32_t>(r);
                        if constexpr (NOUT > 1) out[1][j] = static_cast<uint32_t>(r >> 32);
                    }
                }
            }
            count_fallbacks_warp(a.fallbacks, 2u * __popc(near));
#pragma unroll
            for (int o = 0; o < NOUT; ++o) amax[o] = amax32_lane(out[o]);
        }
    }
}

// The same for the row pass of "both" mode, chunk by chunk: each chunk's
// values are settled (settle_pair on its flagged pairs, or on all four if a
// gate is outside the fast range or a value is huge or infinite -- the
// per-chunk form of the block rules, which is all they need) and written at
// once over the chunk's inputs in the value slots, so only one chunk of
// outputs lives in registers.  Returns the outputs' amax.
template <int OP, int ACT>
__device__ __forceinline__ void block_values_split(const KernelArgs &a, uint8_t *stage, int tile_bytes_,
                                                   const uint32_t (&roff)[4], uint32_t (&amax)[2])
{
    constexpr int NOUT = OpTraits<OP>::kOut;
    constexpr int NIN = OpTraits<OP>::kIn;
    uint32_t acc[2] = {0u, 0u};   // running max of magnitudes (sign bits ignored)
    uint32_t nfb = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t in[3][4];
#pragma unroll
        for (int k = 0; k < NIN; ++k) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + k * tile_bytes_ + roff[c]);
            in[k][0] = v.x;
            in[k][1] = v.y;
            in[k][2] = v.z;
            in[k][3] = v.w;
        }
        uint32_t o4[2][4];
        uint32_t near = 0;   // bit p: pair p of the chunk
        bool far;
        if constexpr (OP == kFwd) {
            far = !gates_fast8(in[0], Gated<ACT>::kMinGate2);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint64_t H = Gated<ACT>::h2(in[0][p], in[1][p]);
                o4[0][p] = pack_bf16x2(f2lo(H), f2hi(H));
                near |= static_cast<uint32_t>(near_mid2(H, Gated<ACT>::kWinH)) << p;
            }
        } else {
            far = !gates_fast8(in[1], Gated<ACT>::kMinGate2);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint64_t DG, DU;
                Gated<ACT>::grads2(in[0][p], in[1][p], in[2][p], DG, DU);
                o4[0][p] = pack_bf16x2(f2lo(DG), f2hi(DG));
                o4[1][p] = pack_bf16x2(f2lo(DU), f2hi(DU));
                near |= static_cast<uint32_t>(near_mid2(DG, Gated<ACT>::kWinDgate) | near_mid2(DU, Gated<ACT>::kWinDup)) << p;
            }
        }
        uint32_t cm[2];
        bool full = false, nanc = false;
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
            cm[o] = hmax_abs2(hmax_abs2(o4[o][0], o4[o][1]), hmax_abs2(o4[o][2], o4[o][3]));
            const uint32_t m = hmax_abs2(cm[o], __byte_perm(cm[o], 0, 0x1032)) & 0x7FFFu;
            full |= huge_amax(m);
            nanc |= nan_amax(m);
        }
        if (__any_sync(0xFFFFFFFFu, near != 0u || far || full || nanc)) {
            if (full || far || nanc) near = 0xFu;
            const void *ta = Gated<ACT>::table_a(a), *tb = Gated<ACT>::table_b(a);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if ((near >> p) & 1u) {
                    // the pair's inputs read again from the stage (still there),
                    // so that the chunk's input registers are free here
                    const uint32_t cj = roff[c];
                    const uint64_t r = settle_pair<OP, ACT>(ta, tb, word_at(stage, cj, p),
                                                            word_at(stage + tile_bytes_, cj, p),
                                                            NIN > 2 ? word_at(stage + 2 * tile_bytes_, cj, p) : 0u, full);
                    o4[0][p] = static_cast<uint32_t>(r);
                    if constexpr (NOUT > 1) o4[1][p] = static_cast<uint32_t>(r >> 32);
                }
            }
            nfb += 2u * __popc(near);
#pragma unroll
            for (int o = 0; o < NOUT; ++o)
                cm[o] = hmax_abs2(hmax_abs2(o4[o][0], o4[o][1]), hmax_abs2(o4[o][2], o4[o][3]));
        }
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
            acc[o] = hmax_abs2(acc[o], cm[o]);
            *reinterpret_cast<uint4 *>(stage + (NIN - NOUT + o) * tile_bytes_ + roff[c]) =
                make_uint4(o4[o][0], o4[o][1], o4[o][2], o4[o][3]);
        }
    }
#pragma unroll
    for (int o = 0; o < NOUT; ++o) amax[o] = hmax_abs2(acc[o], __byte_perm(acc[o], 0, 0x1032)) & 0x7FFFu;
    if (__any_sync(0xFFFFFFFFu, nfb != 0u)) count_fallbacks_warp(a.fallbacks, nfb);
}

// Values already settled (the row pass's outputs in "both" mode, or the
// cast's input), NV slots from `stage`: just load them and take the amax.
template <int NV, bool kAmax = true>
__device__ __forceinline__ void block_settled(const uint8_t *stage, int tile_bytes_, const uint32_t (&roff)[4],
                                              uint32_t (&out)[2][16], uint32_t (&amax)[2])
{
#pragma unroll
    for (int o = 0; o < NV; ++o) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + o * tile_bytes_ + roff[c]);
            out[o][4 * c + 0] = v.x;
            out[o][4 * c + 1] = v.y;
            out[o][4 * c + 2] = v.z;
            out[o][4 * c + 3] = v.w;
        }
        if constexpr (kAmax) amax[o] = amax32_lane(out[o]);
    }
}

// In-place transpose of the warp's 32x32 bf16 sub-tile in one slot: afterwards
// row r of the sub-tile holds column r of the original (rows 0..31 in order).
// ld_addr: this lane's ldmatrix address of unit k (= its row's chunk k);
// st_addr[k]: its stmatrix address of unit k.
__device__ __forceinline__ void transpose_subtile(uint32_t slot, const uint32_t (&roff)[4],
                                                  const uint32_t (&st_off)[4])
{
    uint32_t r[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ldsm_x4_trans(slot + roff[k], r[k]);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) stsm_x4(slot + st_off[k], r[k]);
    __syncwarp();
}

// the lane's 32 bf16 values (16 words) to row `row`, columns c0..c0+31 of h
__device__ __forceinline__ void store_h(const KernelArgs &a, const uint32_t (&v)[16], int64_t row, int64_t c0)
{
    uint16_t *dst = a.h_out + row * a.ld_h + c0;
    if (a.wide_h) {
        const uint32_t lo[8] = {v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]};
        const uint32_t hi[8] = {v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]};
        st_global_v8(dst, lo);
        st_global_v8(dst + 16, hi);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            __stcs(reinterpret_cast<uint4 *>(dst) + j, make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    }
}

// encode the lane's block(s) and store the 32 codes at `q` (16-byte aligned;
// one 256-bit store -- a whole sector -- when `wide` says 32-byte aligned);
// returns the scale bytes in b[o]
template <int NOUT>
__device__ __forceinline__ void store_codes(const uint32_t (&out)[2][16], const uint32_t (&amax)[2],
                                            uint8_t *const (&q)[2], bool live, bool wide, uint32_t (&b)[2])
{
#pragma unroll
    for (int o = 0; o < NOUT; ++o) {
        uint32_t c[8];
        b[o] = encode_block32(out[o], amax[o], c);
        if (live) {
            if (wide) {
                st_global_v8(q[o], c);
            } else {
                __stcs(reinterpret_cast<uint4 *>(q[o]), make_uint4(c[0], c[1], c[2], c[3]));
                __stcs(reinterpret_cast<uint4 *>(q[o]) + 1, make_uint4(c[4], c[5], c[6], c[7]));
            }
        }
    }
}

// The lane's row-scale words of one column tile (NB consecutive 32-row
// blocks: rows r0 + lane + 32 j) in the blocked layout, where the rows of a
// 128-row tile that share r % 32 fill one 16-byte chunk, word (r / 32) % 4:
// the words of consecutive blocks inside one tile go out as one store.  K0 =
// (r0 / 32) % 4; `chunk` is the lane's chunk in the first tile, `stride` the
// bytes between vertically adjacent tiles.
template <int K0, int NB>
__device__ __forceinline__ void store_blocked_words(uint8_t *chunk, int64_t stride, const uint32_t (&w)[NB])
{
#pragma unroll
    for (int p0 = 0; p0 < K0 + NB; p0 += 4) {          // each 128-row tile the band touches
        const int lo = p0 > K0 ? p0 : K0, hi = p0 + 4 < K0 + NB ? p0 + 4 : K0 + NB;
        uint8_t *dst = chunk + (p0 >> 2) * stride + 4 * (lo - p0);
        const uint32_t *v = w + (lo - K0);
        if (hi - lo == 4) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(v[0], v[1], v[2], v[3]);
        } else if (hi - lo == 2 && (lo & 1) == 0) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(v[0], v[1]);
        } else {
            for (int q = 0; q < hi - lo; ++q) reinterpret_cast<uint32_t *>(dst)[q] = v[q];
        }
    }
}

// Row scales of a whole band (rows r0 .. r0 + TM - 1 after any group shift,
// r0 a multiple of 32) in the blocked layout, for the group's gsize column
// tiles: per tile and output, the lane reads its TM / 32 words from the
// group's buffer and stores them chunk by chunk (s_row 16-byte aligned).
template <int NOUT, int TM, int G>
__device__ __forceinline__ void flush_blocked_band(const KernelArgs &a, const uint8_t *gbuf, int64_t r0,
                                                   int64_t blk0, int gsize, int lane)
{
    constexpr int NB = TM / 32;
    const int k0 = static_cast<int>((r0 >> 5) & 3);
    const int64_t stride = a.srow_tiles_c * 512;
    for (int t = 0; t < gsize; ++t) {
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
            const uint8_t *src = gbuf + o * scale_group_bytes<TM, G>() + 4 * G * lane + 4 * t;
            uint32_t w[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) w[j] = *reinterpret_cast<const uint32_t *>(src + 4 * G * 32 * j);
            uint8_t *chunk = a.s_row[o] + ((r0 >> 7) * a.srow_tiles_c + (blk0 >> 2) + t) * 512 + 16 * lane;
            switch (k0) {
            case 0: store_blocked_words<0, NB>(chunk, stride, w); break;
            case 1: store_blocked_words<1, NB>(chunk, stride, w); break;
            case 2: store_blocked_words<2, NB>(chunk, stride, w); break;
            default: store_blocked_words<3, NB>(chunk, stride, w); break;
            }
        }
    }
}

// Row scales of one finished group of column tiles (tiles 0..gsize-1 of group
// ug in row band tr), from its shared-memory buffer (4 G bytes a row) to s_row,
// by the whole producer warp.  Row-major: one 4G-byte store per row where the
// group is whole and rows are aligned (`wide`), single bytes otherwise.
// Blocked (plain, per group or per expert): whole bands whose 32-row blocks
// share one group shift go out chunk by chunk (flush_blocked_band); a ragged
// last band, or one that a group boundary with a new shift crosses, row by
// row.  The per-group layouts write nothing if the group ends were found
// invalid.  (The producer issues the next tile's loads only after this, so
// its instruction count bounds how far it can run ahead.)
template <int NOUT, int TM, int G, bool GRP>
__device__ __forceinline__ void flush_row_scales(const KernelArgs &a, const uint8_t *gbuf, int64_t tr, int64_t ug,
                                                 int gsize, int lane, const int32_t *gtab, int &hint)
{
    constexpr int kBlocks = TM / 32;
    const int64_t row0 = tr * TM;
    const int64_t blk0 = ug * 4 * G;
    const int64_t nblk = a.N >> 5;
    if (GRP || a.blocked) {
        int32_t mine = 0;     // lane j < kBlocks: the row shift of the band's block j
        // the plain layout with one column tile a group and bands that
        // straddle 128-row tiles (the rowwise cast's 192 rows) measured
        // faster row by row (521 against 540 us at 131072 x 8192; the "both"
        // cast, four tiles a group, 678 against 803 the other way)
        bool band = row0 + TM <= a.M && (GRP || TM % 128 == 0 || G > 1);
#pragma unroll
        for (int o = 0; o < NOUT; ++o) band &= (reinterpret_cast<uintptr_t>(a.s_row[o]) & 15u) == 0;
        if constexpr (GRP) {
            if (a.group_end != nullptr && gtab[3 * kMaxGroups] == 0) return;
            const int64_t brow0 = row0 + 32 * lane;
            mine = (lane < kBlocks && brow0 < a.M) ? static_cast<int32_t>(group_shift(a, gtab, brow0, hint).r) : 0;
        }
        const int32_t rsh0 = __shfl_sync(0xFFFFFFFFu, mine, 0);
        if (__all_sync(0xFFFFFFFFu, band && (lane >= kBlocks || mine == rsh0))) {
            flush_blocked_band<NOUT, TM, G>(a, gbuf, row0 + rsh0, blk0, gsize, lane);
            return;
        }
#pragma unroll
        for (int j = 0; j < kBlocks; ++j) {
            const int32_t rsh = __shfl_sync(0xFFFFFFFFu, mine, j);
            const int i = lane + 32 * j;
            const int64_t row = row0 + i;
            if (row >= a.M) continue;
#pragma unroll
            for (int o = 0; o < NOUT; ++o) {
                const uint8_t *src = gbuf + o * scale_group_bytes<TM, G>() + 4 * G * i;
                // a tile's four blocks of a row are contiguous in the blocked
                // layout (padding blocks of the last tile come out as 0)
                for (int t = 0; t < gsize; ++t)
                    *reinterpret_cast<uint32_t *>(a.s_row[o] + blocked_offset(row + rsh, blk0 + 4 * t, a.srow_tiles_c)) =
                        *reinterpret_cast<const uint32_t *>(src + 4 * t);
            }
        }
        return;
    }
    const bool whole = a.wide_srow != 0 && gsize == G && blk0 + 4 * G <= nblk;
    for (int i = lane; i < TM; i += 32) {
        const int64_t row = row0 + i;
        if (row >= a.M) break;
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
            const uint8_t *src = gbuf + o * scale_group_bytes<TM, G>() + 4 * G * i;
            uint8_t *dst = a.s_row[o] + row * a.ld_srow + blk0;
            if (whole) {
                if constexpr (G == 4)
                    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
                else if constexpr (G == 2)
                    *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(src);
                else
                    *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(src);
            } else {
                for (int j = 0; j < 4 * gsize; ++j)
                    if (blk0 + j < nblk) dst[j] = src[j];
            }
        }
    }
}

// This CTA's tiles.  Column tiles are taken in groups of G consecutive ones
// of a row band ("super-tiles" u = blockIdx.x, + gridDim.x, ...), tile by
// tile; the walk keeps the row band tr, the group ug, the tile i within it,
// the pipeline slot (stage, phase parity) and the group's row-scale buffer
// slot (group ordinal % (STAGES + 1)), advanced without divisions.  32-bit
// counters (the host rejects tile counts that do not fit): they are live
// across the whole tile loop, so every register they save counts.
template <int STAGES, int G>
struct TileWalk {
    int32_t u, tr, ug, step_r, step_c, tiles_g, tiles_n;
    int i, gsize, s, gslot;
    uint32_t ph;
    __device__ __forceinline__ explicit TileWalk(int64_t n_tiles_n)
        : u(static_cast<int32_t>(blockIdx.x)), tiles_n(static_cast<int32_t>(n_tiles_n)), i(0), s(0), gslot(0), ph(0)
    {
        tiles_g = (tiles_n + G - 1) / G;
        tr = u / tiles_g;
        ug = u - tr * tiles_g;
        step_r = static_cast<int32_t>(gridDim.x) / tiles_g;
        step_c = static_cast<int32_t>(gridDim.x) - step_r * tiles_g;
        gsize = min(G, tiles_n - ug * G);
    }
    __device__ __forceinline__ int64_t tc() const { return static_cast<int64_t>(ug) * G + i; }
    __device__ __forceinline__ bool last_in_group() const { return i + 1 == gsize; }
    __device__ __forceinline__ void next()
    {
        if (++i == gsize) {
            i = 0;
            u += gridDim.x;
            tr += step_r;
            ug += step_c;
            if (ug >= tiles_g) {
                ug -= tiles_g;
                ++tr;
            }
            gsize = min(G, tiles_n - ug * G);
            if (++gslot == STAGES + 1) gslot = 0;
        }
        if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// ------------------------------------------------------------------ kernel
template <int OP, int MODE, int TM, int STAGES, int CTAS, int G, int ACT, bool GRP>
__global__ void __launch_bounds__((warps_of<TM>() + 1) * 32, CTAS)
    mxfp8_tile_kernel(const __grid_constant__ CUtensorMap tm0,
                      const __grid_constant__ CUtensorMap tm1,
                      const __grid_constant__ CUtensorMap tm2, const KernelArgs a)
{
    constexpr int NIN = OpTraits<OP>::kIn;
    constexpr int NOUT = OpTraits<OP>::kOut;
    constexpr int kWarps = warps_of<TM>();
    constexpr int kTileM = TM;
    constexpr int kBoxBytes = TM * kBoxN * 2;
    constexpr int kTileBytes = tile_bytes<TM>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // row-scale buffers [slot][output]: a group of column tiles uses slot
    // (group ordinal % (STAGES + 1)), so the producer can write a finished
    // group's scales out after refilling the stage of its last tile
    uint8_t *sbuf0 = smem + STAGES * NIN * kTileBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf0 + (STAGES + 1) * NOUT * scale_group_bytes<TM, G>());
    const uint32_t smem_base = smem_u32(smem);
    // a full and an empty barrier per stage and part: the SwiGLU fused ops
    // split a stage into its two 64-column halves, so the warps reading one
    // TMA box free it without waiting for the other half (measured: faster
    // for them, slower for the compute-bound GEGLU and no gain for the cast)
    constexpr int kParts = (ACT == kSilu && OP != kQuant) ? 2 : 1;
    constexpr int kBoxesPerPart = 2 / kParts;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + 2 * STAGES);
    // per-group layouts (GRP instantiations only): the group table
    int32_t *gtab = reinterpret_cast<int32_t *>(bars + 4 * STAGES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            for (int h = 0; h < kParts; ++h) {
                mbar_init(full0 + 8 * (2 * s + h), 1);
                mbar_init(empty0 + 8 * (2 * s + h), kWarps / kParts);
            }
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if constexpr (GRP) {
        static_assert(STAGES <= kMaxColStages && TM / 32 <= kMaxColBlocks, "column-shift slots");
        if (a.group_end != nullptr && warp == 0) {
            const bool ok = build_group_table(a.group_end, a.num_groups, a.M, gtab, lane);
            if (lane == 0) {
                gtab[3 * kMaxGroups] = ok ? 1 : 0;
                if (!ok && blockIdx.x == 0) atomicOr(a.status, kStatusBadGroups);
            }
        }
    }
    if constexpr (ACT == kGelu && OP != kQuant) gelu_tail_fill<OP == kFwd>(a.gelu_tail);
    __syncthreads();

    const int64_t tiles_n = a.tiles_n;
    const int64_t num_super = (a.num_tiles / tiles_n) * ((tiles_n + G - 1) / G);   // groups of column tiles

    // ------------------------------------------------------- producer warp
    // Lane 0 streams the tiles in; once a stage has been refilled, the whole
    // warp writes the row scales of the tile that occupied it out of their
    // buffer (and those of the last tiles at the end).
    if (warp == kWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm0);
            if (NIN > 1) prefetch_tensormap(&tm1);
            if (NIN > 2) prefetch_tensormap(&tm2);
        }
        int it = 0;
        int ghint = 0;     // group of this lane's last row-scale lookup
        int chint = 0;     // the same for the column shifts
        bool failed = false;
        TileWalk<STAGES, G> done(tiles_n);   // the oldest tile not yet recycled
        for (TileWalk<STAGES, G> w(tiles_n); w.u < num_super; w.next(), ++it) {
            const int s = w.s;
            // per-group column scales: lane j < TM / 32 finds the shift of the
            // tile's 32-row block j, handed to the column pass through the
            // stage's slots below
            int32_t csh_c = 0, csh_r = 0;
            if constexpr (GRP && (MODE & kCol)) {
                const int64_t brow = static_cast<int64_t>(w.tr) * kTileM + 32 * lane;
                if (lane < kTileM / 32 && brow < a.M) {
                    const GroupShift gs = group_shift(a, gtab, brow, chint);
                    csh_c = static_cast<int32_t>(gs.c);
                    csh_r = static_cast<int32_t>(gs.crow);
                }
            }
#pragma unroll
            for (int h = 0; h < kParts; ++h) {
                if (it >= STAGES) {
                    bool ok = lane == 0 ? mbar_wait_bounded(empty0 + 8 * (2 * s + h), w.ph ^ 1u, a.wait_limit) : true;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok) {
                        if (lane == 0) {
                            atomicOr(a.status, kStatusProducerWait);
                            // part 0 of this tile is already in flight: wait for it
                            if (h == 1 && !mbar_wait_bounded(full0 + 8 * (2 * s), w.ph, a.wait_limit))
                                atomicOr(a.status, kStatusDrainWait);
                        }
                        failed = true;
                        break;
                    }
                }
                if constexpr (GRP && (MODE & kCol)) {
                    // the part's copy of the shifts, then the arrive below
                    // releases them to the part's consumers
                    if (lane < kTileM / 32) {
                        gtab[col_shift_word(s, h, lane)] = csh_c;
                        gtab[col_shift_word(s, h, lane) + 1] = csh_r;
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    const int32_t r0 = w.tr * kTileM;
                    const uint32_t bar = full0 + 8 * (2 * s + h);
                    mbar_expect_tx(bar, NIN * kBoxesPerPart * kBoxBytes);
#pragma unroll
                    for (int x = 0; x < kBoxesPerPart; ++x) {
                        const int box = h * kBoxesPerPart + x;
                        const int32_t c0 = static_cast<int32_t>(w.tc() * kTileN) + box * kBoxN;
                        const uint32_t dst = smem_base + static_cast<uint32_t>(s * NIN) * kTileBytes + box * kBoxBytes;
                        tma_load_2d(dst, &tm0, c0, r0, bar);
                        if (NIN > 1) tma_load_2d(dst + kTileBytes, &tm1, c0, r0, bar);
                        if (NIN > 2) tma_load_2d(dst + 2 * kTileBytes, &tm2, c0, r0, bar);
                    }
                }
            }
            if (failed) break;
            if (it >= STAGES) {
                // tile it - STAGES is finished (its stage was free); if it ends
                // its group, the group's slot is written again only by a
                // group starting at tile it + 1 or later, loaded after this
                if constexpr (MODE & kRow) {
                    if (done.last_in_group())
                        flush_row_scales<NOUT, TM, G, GRP>(a, sbuf0 + done.gslot * NOUT * scale_group_bytes<TM, G>(), done.tr,
                                                      done.ug, done.gsize, lane, gtab, ghint);
                }
                done.next();
            }
            __syncwarp();
        }
        // the last tiles: wait (bounded) until the consumers have finished
        // each, then write its row scales; after a failure, only wait for the
        // loads still in flight
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
            const int s = j % STAGES;
            const uint32_t ph = static_cast<uint32_t>(j / STAGES) & 1u;
            bool ok;
            if (failed) {
                // every part of every issued tile
                for (int h = 0; h < kParts; ++h) {
                    ok = lane == 0 ? mbar_wait_bounded(full0 + 8 * (2 * s + h), ph, a.wait_limit) : true;
                    if (!ok && lane == 0) atomicOr(a.status, kStatusDrainWait);
                }
                continue;
            }
            ok = lane == 0 ? (mbar_wait_bounded(empty0 + 8 * (2 * s), ph, a.wait_limit) &&
                              (kParts == 1 || mbar_wait_bounded(empty0 + 8 * (2 * s + 1), ph, a.wait_limit)))
                           : true;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicOr(a.status, kStatusProducerWait);
                break;
            }
            if constexpr (MODE & kRow) {
                if (done.last_in_group() || j + 1 == it)
                    flush_row_scales<NOUT, TM, G, GRP>(a, sbuf0 + done.gslot * NOUT * scale_group_bytes<TM, G>(), done.tr,
                                                  done.ug, done.i + 1, lane, gtab, ghint);
            }
            done.next();
        }
        return;
    }

    // ------------------------------------------------------- consumer warps
    const uint32_t srb = static_cast<uint32_t>(warp >> 2);        // sub-tile row block
    const uint32_t scb = static_cast<uint32_t>(warp & 3);         // sub-tile column block
    const uint32_t box_off = (scb >> 1) * kBoxBytes;              // which 64-column box
    const uint32_t chunk0 = (scb & 1) * 4;                        // first 16-byte chunk in it
    // this lane's sub-tile row: chunk offsets within a slot (row pass reads,
    // col pass reads of the transposed rows, ldmatrix addresses of unit k)
    const uint32_t myrow = kSub * srb + static_cast<uint32_t>(lane);
    uint32_t roff[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) roff[c] = box_off + swz(myrow, chunk0 + c);
    // stmatrix address of unit k: matrix m = lane/8 -> chunk m of row 8k + lane%8
    uint32_t st_off[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        st_off[k] = box_off + swz(kSub * srb + 8u * k + (static_cast<uint32_t>(lane) & 7u),
                                  chunk0 + (static_cast<uint32_t>(lane) >> 3));

    constexpr bool kSplit = (MODE == kBoth) && (OP != kQuant);  // values handed row -> col pass
    // the forward's col mode evaluates h row by row (lanes own rows, as in
    // the row pass) into the up slot and transposes that one slot, rather
    // than transposing gate and up and evaluating column by column: fewer
    // shared-memory round trips (measured faster for the forward, SwiGLU
    // 825 -> 809 us and GEGLU 1002 -> 943 at 131072 x 8192, and slower for
    // the backward, 1362 -> 1462 us, and for the per-group forward, 879 ->
    // 934 us)
    constexpr bool kVF = (MODE == kCol) && (OP == kFwd) && !GRP;
    // generic writes into the stage (the values handed to the col pass, the
    // transposes, the forward rare path's results)
    constexpr bool kWrites = kSplit || (MODE & kCol) || OP == kFwd;
    for (TileWalk<STAGES, G> w(tiles_n); w.u < num_super; w.next()) {
        const int s = w.s;
        const uint32_t part = kParts == 2 ? (scb >> 1) : 0u;     // the half this warp reads
        const bool fail = __any_sync(0xFFFFFFFFu, !mbar_wait_bounded(full0 + 8 * (2 * s + part), w.ph, a.wait_limit));
        if (fail) {
            if (lane == 0) atomicOr(a.status, kStatusConsumerWait);
            return;
        }
        const int64_t r0 = static_cast<int64_t>(w.tr) * kTileM + kSub * srb;   // sub-tile origin
        const int64_t c0 = w.tc() * kTileN + kSub * scb;
        const uint32_t stage = smem_base + static_cast<uint32_t>(s * NIN) * kTileBytes;
        const uint8_t *stage_ptr = smem + static_cast<size_t>(s * NIN) * kTileBytes;

        if constexpr (MODE & kRow) {
            const int64_t grow = r0 + lane;
            const bool live = grow < a.M && c0 < a.N;
            uint32_t b[2];
            if constexpr (kSplit && OP == kBwd && ACT != kGeluPoly) {
                // values settled chunk by chunk into the value slots (which
                // the col pass then transposes), encoded from there: only one
                // chunk of the two outputs lives in registers (measured: a
                // gain for the backward, a loss for the forward)
                uint32_t amax[2];
                block_values_split<OP, ACT>(a, const_cast<uint8_t *>(stage_ptr), kTileBytes, roff, amax);
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    uint32_t v[2][16], am[2];
                    block_settled<1, false>(stage_ptr + (NIN - NOUT + o) * kTileBytes, kTileBytes, roff, v, am);
                    uint8_t *q[2] = {a.q_row[o] + grow * a.ld_qrow + c0, nullptr};
                    uint32_t bb[2];
                    const uint32_t amx[2] = {amax[o], 0u};
                    store_codes<1>(v, amx, q, live, a.wide_row != 0, bb);
                    b[o] = bb[0];
                }
                __syncwarp();
            } else {
                uint32_t out[2][16], amax[2];
                block_values<OP, ACT, OP == kFwd && MODE == kBoth>(a, stage_ptr, kTileBytes, roff, out, amax);
                if constexpr (OP == kFwd) {
                    // the activation itself, for callers that keep it in bf16
                    // (per-lane stores: staging it for a TMA store measured
                    // slower, 1269 against 1253 us at 131072 x 8192)
                    if (a.h_out != nullptr && live) store_h(a, out[0], grow, c0);
                }
                uint8_t *q[2];
#pragma unroll
                for (int o = 0; o < NOUT; ++o) q[o] = a.q_row[o] + grow * a.ld_qrow + c0;
                store_codes<NOUT>(out, amax, q, live, a.wide_row != 0, b);
                if constexpr (kSplit) {
                    // the values the col pass encodes, over inputs no longer needed
#pragma unroll
                    for (int o = 0; o < NOUT; ++o)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4 *>(const_cast<uint8_t *>(stage_ptr) +
                                                       (NIN - NOUT + o) * kTileBytes + roff[c]) =
                                make_uint4(out[o][4 * c], out[o][4 * c + 1], out[o][4 * c + 2], out[o][4 * c + 3]);
                    __syncwarp();
                }
            }
            // scale bytes to the group's buffer: row (32 srb + lane), block 4 i + scb
            uint8_t *sb = sbuf0 + w.gslot * NOUT * scale_group_bytes<TM, G>() + 4 * G * myrow + 4 * w.i + scb;
#pragma unroll
            for (int o = 0; o < NOUT; ++o) sb[o * scale_group_bytes<TM, G>()] = static_cast<uint8_t>(b[o]);
        }

        if constexpr (MODE & kCol) {
            // transpose the slots the col pass reads: the cast's input, the
            // row pass's values ("both"), the forward's values evaluated just
            // below ("col"), or the backward's inputs ("col")
            if constexpr (kVF) {
                uint32_t vo[2][16], am[2];
                block_values<OP, ACT>(a, stage_ptr, kTileBytes, roff, vo, am);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(const_cast<uint8_t *>(stage_ptr) + (NIN - NOUT) * kTileBytes + roff[c]) =
                        make_uint4(vo[0][4 * c], vo[0][4 * c + 1], vo[0][4 * c + 2], vo[0][4 * c + 3]);
                __syncwarp();
            }
            constexpr int kFirst = (kSplit || kVF) ? NIN - NOUT : 0;
            constexpr int kCount = (kSplit || kVF) ? NOUT : NIN;
#pragma unroll
            for (int k = 0; k < kCount; ++k)
                transpose_subtile(stage + static_cast<uint32_t>((kFirst + k) * kTileBytes), roff, st_off);
            const int64_t gcol = c0 + lane;
            const bool live = r0 < a.M && gcol < a.N;
            uint32_t out[2][16], amax[2];
            if constexpr (kSplit || kVF || OP == kQuant)
                block_settled<NOUT>(stage_ptr + kFirst * kTileBytes, kTileBytes, roff, out, amax);
            else
                block_values<OP, ACT, false, false>(a, stage_ptr, kTileBytes, roff, out, amax);
            int64_t grp = 0, rin = r0;
            if (a.group_stride != 0) {  // 3D: per-expert column-major output
                grp = r0 / a.group_rows;
                rin = r0 - grp * a.group_rows;
            }
            uint8_t *q[2];
#pragma unroll
            for (int o = 0; o < NOUT; ++o) q[o] = a.q_col[o] + grp * a.group_stride + gcol * a.ld_qcol + rin;
            uint32_t b[2];
            store_codes<NOUT>(out, amax, q, live, a.wide_col != 0, b);
            if constexpr (GRP) {
                // per-group layouts (the same shift for the whole warp)
                const bool ok = a.group_end == nullptr || gtab[3 * kMaxGroups] != 0;
                // the block's shifts, found by the producer when it loaded
                // the tile (a lookup here, in every warp's tile loop, cost
                // 4-8 % of the kernel)
                const int32_t *csh = gtab + col_shift_word(s, part, static_cast<int>(srb));
                if (live && ok) {
                    const int64_t off = blocked_offset(gcol + csh[1], (r0 >> 5) + csh[0], a.scol_tiles_c);
#pragma unroll
                    for (int o = 0; o < NOUT; ++o) a.s_col[o][off] = static_cast<uint8_t>(b[o]);
                }
            } else if (live) {
                const int64_t off = a.blocked ? blocked_offset(gcol, r0 >> 5, a.scol_tiles_c) : (r0 >> 5) * a.ld_scol + gcol;
#pragma unroll
                for (int o = 0; o < NOUT; ++o) a.s_col[o][off] = static_cast<uint8_t>(b[o]);
            }
        }

        if constexpr (kWrites) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * (2 * s + part));
    }
}

}  // namespace mx
