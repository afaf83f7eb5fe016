// kernel.cuh -- the persistent tile kernel shared by every entry point.
//
// One CTA per SM: 16 consumer warps and one producer warp.  The producer's
// lane 0 streams the input tiles (128 rows x 128 bf16 columns per tensor, as
// two 64-column boxes with the 128-byte swizzle) into a ring of shared-memory
// stages with TMA; each stage has a "full" mbarrier (transaction bytes) and
// an "empty" mbarrier (one arrive per consumer warp).
//
// Consumer warp w owns the 32 x 32 sub-tile (row block w/4, column block w%4)
// of every tile, so no two warps ever share data and the only
// synchronisation inside a tile is __syncwarp:
//   row pass: four iterations of 8 rows; a lane holds one 16-byte chunk
//             (8 elements) of a row, four consecutive lanes one 1x32 block.
//             The element op runs on the chunk, the block amax takes two
//             shuffles, each lane stores its 8 E4M3 codes (the four lanes: 32
//             contiguous bytes).
//   col pass: four 32-row x 8-column units; ldmatrix.trans gives four lanes
//             one column of a unit, which is encoded colwise; stmatrix moves
//             the codes into a warp-private staging buffer, column by column,
//             and each lane stores one column's 32 codes (32 contiguous bytes
//             of the column-major output).
// In "both" mode the row pass writes the bf16 element values back into the
// stage (over an input it no longer needs), so both scale sets come from one
// read of the inputs.  In "col" mode the element op runs directly on the
// transposed fragments.
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

// Tile height and pipeline depth per instantiation: more warps hide more
// latency where the registers allow it (the cast alone needs few).
template <int OP, int MODE>
struct Tuning {
    static constexpr int kTM = OP == kQuant ? 224 : ((OP == kFwd && MODE != kBoth) ? 192 : 128);
    static_assert((kTM / 32) * 4 + 1 <= 32, "at most 1024 threads per CTA");
    static constexpr int kStages = OP == kQuant ? 3 : 2 + (OP == kFwd && MODE == kBoth);
};

template <int TM>
__host__ __device__ constexpr int warps_of() { return (TM / kSub) * (kTileN / kSub); }

template <int TM>
__host__ __device__ constexpr int tile_bytes() { return TM * kTileN * 2; }

// shared memory: 1 KB alignment slack, the stages, the per-warp colwise
// staging buffers (1 KB per output), the mbarriers
template <int OP, int TM, int STAGES>
constexpr size_t smem_bytes()
{
    return 1024 + static_cast<size_t>(STAGES) * OpTraits<OP>::kIn * tile_bytes<TM>() +
           static_cast<size_t>(warps_of<TM>()) * OpTraits<OP>::kOut * 1024 + 2 * STAGES * 8;
}

// ------------------------------------------------------- element operation
// Fast element op on 8 elements (4 packed bf16x2 words per input) into
// out[o][4] (packed bf16x2 words).  With kKeep the fp32 pairs are kept in
// hv[o][4] for a later look (returns 0); without it the pairs (bit p:
// elements 2p and 2p+1) holding a value near a 0x60/0x61 rounding midpoint
// are returned.
template <int OP, bool kKeep>
__device__ __forceinline__ uint32_t elements8(const uint32_t (&in)[3][4], uint32_t (&out)[2][4],
                                              uint64_t (&hv)[2][4])
{
    uint32_t near = 0;
    if constexpr (OP == kQuant) {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[0][i] = in[0][i];
    } else if constexpr (OP == kFwd) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint64_t H = swiglu_h2(in[0][p], in[1][p]);
            out[0][p] = pack_bf16x2(f2lo(H), f2hi(H));
            if constexpr (kKeep) hv[0][p] = H;
            else near |= static_cast<uint32_t>(near_mid2(H, kNearH)) << p;
        }
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint64_t DG, DU;
            swiglu_grads2(in[0][p], in[1][p], in[2][p], DG, DU);
            out[0][p] = pack_bf16x2(f2lo(DG), f2hi(DG));
            out[1][p] = pack_bf16x2(f2lo(DU), f2hi(DU));
            if constexpr (kKeep) {
                hv[0][p] = DG;
                hv[1][p] = DU;
            } else {
                near |= static_cast<uint32_t>(near_mid2(DG, kNearDgate) | near_mid2(DU, kNearDup)) << p;
            }
        }
    }
    return near;
}

__device__ __forceinline__ uint32_t bf16_bits(float v) { return pack_bf16x2(v, 0.0f) & 0xFFFFu; }

__device__ __forceinline__ void set_half16(uint32_t &w, int hi, uint32_t b)
{
    w = hi ? ((w & 0xFFFFu) | (b << 16)) : ((w & 0xFFFF0000u) | b);
}

// exact value(s) of element e (0..7) from the inputs in registers
template <int OP>
__device__ __forceinline__ void exact_element(const KernelArgs &a, const uint32_t (&in)[3][4], int e,
                                              uint32_t (&out)[2][4])
{
    const int p = e >> 1, hi = e & 1;
    const float x0 = hi ? bf16hi(in[0][p]) : bf16lo(in[0][p]);
    const float x1 = hi ? bf16hi(in[1][p]) : bf16lo(in[1][p]);
    if constexpr (OP == kFwd) {
        set_half16(out[0][p], hi, bf16_bits(swiglu_h_exact(a.sig2_table, x0, x1)));
    } else if constexpr (OP == kBwd) {
        const float x2 = hi ? bf16hi(in[2][p]) : bf16lo(in[2][p]);
        const float2 x = swiglu_grads_exact(a.sig2_table, x0, x1, x2);
        set_half16(out[0][p], hi, bf16_bits(x.x));
        set_half16(out[1][p], hi, bf16_bits(x.y));
    }
}

// Settle a lane's fast values (row pass; col pass of "col" mode): exact
// recomputation of all 8 elements if a gate is outside the fast range or the
// block amax is huge or not finite; otherwise of the pairs near a 0x60/0x61
// rounding midpoint.  With kKeep the midpoint test runs only in blocks whose
// fast amax has mantissa 0x60 or 0x61 -- a scale can move nowhere else --
// on the kept fp32 values; without it `near` holds the test's result for
// every pair (needed when the values also feed the other direction's
// blocks).  amax[o] is kept current.  Warp-uniform control flow around every
// shuffle.
template <int OP, bool kKeep>
__device__ __forceinline__ void settle(const KernelArgs &a, const uint32_t (&in)[3][4],
                                       uint32_t (&out)[2][4], uint32_t (&amax)[2], uint32_t near,
                                       const uint64_t (&hv)[2][4])
{
    constexpr int NOUT = OpTraits<OP>::kOut;
    constexpr int kGate = (OP == kFwd) ? 0 : 1;
    bool full = !gates_fast8(in[kGate]);
#pragma unroll
    for (int o = 0; o < NOUT; ++o) full |= amax[o] >= kHugeAmax;
    if constexpr (kKeep) {
        bool risk = false;
#pragma unroll
        for (int o = 0; o < NOUT; ++o) risk |= scale_at_risk(amax[o]);
        if (!__any_sync(0xFFFFFFFFu, full || risk)) return;
        if (risk) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                bool n = false;
#pragma unroll
                for (int o = 0; o < NOUT; ++o)
                    n |= scale_at_risk(amax[o]) &&
                         near_mid2(hv[o][p], (OP == kFwd) ? kNearH : (o == 0 ? kNearDgate : kNearDup));
                near |= static_cast<uint32_t>(n) << p;
            }
        }
    }
    if (full) near = 0xFu;
    if (__any_sync(0xFFFFFFFFu, near != 0u)) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            if ((near >> p) & 1u) {
                exact_element<OP>(a, in, 2 * p, out);
                exact_element<OP>(a, in, 2 * p + 1, out);
            }
        }
        count_fallbacks_warp(a.fallbacks, 2u * __popc(near));
#pragma unroll
        for (int o = 0; o < NOUT; ++o) amax[o] = amax32_lanes4(out[o]);
    }
}

// ------------------------------------------------------------------ kernel
template <int OP, int MODE, int TM, int STAGES>
__global__ void __launch_bounds__((warps_of<TM>() + 1) * 32, 1)
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
    uint8_t *staging = smem + STAGES * NIN * kTileBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + kWarps * NOUT * 1024);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kWarps);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    const int64_t num_tiles = a.num_tiles;
    const int64_t tiles_n = a.tiles_n;

    // ------------------------------------------------------- producer warp
    if (warp == kWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm0);
            if (NIN > 1) prefetch_tensormap(&tm1);
            if (NIN > 2) prefetch_tensormap(&tm2);
            int it = 0;
            bool failed = false;
            for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
                if (it >= STAGES && !mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, a.wait_limit)) {
                    atomicOr(a.status, kStatusProducerWait);
                    failed = true;
                    break;
                }
                const int32_t r0 = static_cast<int32_t>((t / tiles_n) * kTileM);
                const int32_t c0 = static_cast<int32_t>((t % tiles_n) * kTileN);
                const uint32_t bar = full0 + 8 * s;
                const uint32_t dst = smem_base + static_cast<uint32_t>(s * NIN) * kTileBytes;
                mbar_expect_tx(bar, NIN * kTileBytes);
                tma_load_2d(dst, &tm0, c0, r0, bar);
                tma_load_2d(dst + kBoxBytes, &tm0, c0 + kBoxN, r0, bar);
                if (NIN > 1) {
                    tma_load_2d(dst + kTileBytes, &tm1, c0, r0, bar);
                    tma_load_2d(dst + kTileBytes + kBoxBytes, &tm1, c0 + kBoxN, r0, bar);
                }
                if (NIN > 2) {
                    tma_load_2d(dst + 2 * kTileBytes, &tm2, c0, r0, bar);
                    tma_load_2d(dst + 2 * kTileBytes + kBoxBytes, &tm2, c0 + kBoxN, r0, bar);
                }
            }
            if (failed) {
                // wait (bounded) for every load still in flight before leaving
                for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j) {
                    const uint32_t ph = static_cast<uint32_t>(j / STAGES) & 1u;
                    if (!mbar_wait_bounded(full0 + 8 * (j % STAGES), ph, a.wait_limit))
                        atomicOr(a.status, kStatusDrainWait);
                }
            }
        }
        return;
    }

    // ------------------------------------------------------- consumer warps
    const uint32_t srb = static_cast<uint32_t>(warp >> 2);        // sub-tile row block
    const uint32_t scb = static_cast<uint32_t>(warp & 3);         // sub-tile column block
    const uint32_t box_off = (scb >> 1) * kBoxBytes;              // which 64-column box
    const uint32_t chunk0 = (scb & 1) * 4;                        // first 16-byte chunk in it
    const uint32_t q = static_cast<uint32_t>(lane & 3);
    // row pass: lane -> row 8i + perm(lane/4), chunk chunk0 + lane%4; the
    // permutation puts rows r and r+4 in one 8-lane phase (conflict-free
    // with the 128-byte swizzle)
    const uint32_t rl = static_cast<uint32_t>(lane >> 2);
    const uint32_t rperm = ((rl & 1u) << 2) | (rl >> 1);
    uint8_t *stg = staging + warp * NOUT * 1024;   // this warp's colwise staging

    constexpr bool kSplit = (MODE == kBoth) && (OP != kQuant);  // values handed row -> col pass
    constexpr bool kKeep = !kSplit;   // midpoint test deferred to risky blocks
    constexpr int kUnroll = (OP == kQuant) ? 4 : 1;  // the cast alone: unroll for ILP
    int it = 0;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
        const bool fail = __any_sync(0xFFFFFFFFu, !mbar_wait_bounded(full0 + 8 * s, ph, a.wait_limit));
        if (fail) {
            if (lane == 0) atomicOr(a.status, kStatusConsumerWait);
            return;
        }
        const int64_t r0 = (t / tiles_n) * kTileM + kSub * srb;   // sub-tile origin
        const int64_t c0 = (t % tiles_n) * kTileN + kSub * scb;
        const uint32_t stage = smem_base + static_cast<uint32_t>(s * NIN) * kTileBytes + box_off;
        uint8_t *stage_ptr = smem + static_cast<size_t>(s * NIN) * kTileBytes + box_off;

        if constexpr (MODE & kRow) {
            // this lane's rows are r0 + 8i + rperm; all addressing is set up
            // once per tile
            const int64_t gcol = c0 + 8 * q;
            const int64_t grow0 = r0 + rperm;
            const int64_t left64 = a.M - grow0;
            const int rows_left = left64 > 32 ? 32 : static_cast<int>(left64 < 0 ? 0 : left64);
            const bool col_ok = gcol < a.N;
            uint8_t *qp[2];
            uint8_t *sp[2];
#pragma unroll
            for (int o = 0; o < NOUT; ++o) {
                qp[o] = a.q_row[o] + grow0 * a.ld_qrow + gcol;
                sp[o] = a.s_row[o] + grow0 * a.ld_srow + (gcol >> 5);
            }
            const int64_t qstep = 8 * a.ld_qrow, sstep = 8 * a.ld_srow;
#pragma unroll kUnroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t row = kSub * srb + 8u * i + rperm;
                const uint32_t off = swz(row, chunk0 + q);
                uint32_t in[3][4];
                uint32_t out[2][4];
                uint64_t hv[2][4];
#pragma unroll
                for (int k = 0; k < NIN; ++k) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(stage_ptr + k * kTileBytes + off);
                    in[k][0] = v.x;
                    in[k][1] = v.y;
                    in[k][2] = v.z;
                    in[k][3] = v.w;
                }
                const uint32_t near = elements8<OP, kKeep>(in, out, hv);
                uint32_t amax[2];
#pragma unroll
                for (int o = 0; o < NOUT; ++o) amax[o] = amax32_lanes4(out[o]);
                if constexpr (OP != kQuant) settle<OP, kKeep>(a, in, out, amax, near, hv);
                const bool live = col_ok && (8 * i < rows_left);
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    uint32_t w0, w1;
                    const uint32_t sc = encode_block8(out[o], amax[o], w0, w1);
                    if (live) {
                        __stcs(reinterpret_cast<uint2 *>(qp[o]), make_uint2(w0, w1));
                        if (q == 0) *sp[o] = static_cast<uint8_t>(sc);
                    }
                    qp[o] += qstep;
                    sp[o] += sstep;
                    if constexpr (kSplit) {
                        *reinterpret_cast<uint4 *>(stage_ptr + (NIN - NOUT + o) * kTileBytes + off) =
                            make_uint4(out[o][0], out[o][1], out[o][2], out[o][3]);
                    }
                }
            }
            if constexpr (kSplit) __syncwarp();
        }

        if constexpr (MODE & kCol) {
            // element values for the col pass: quant reads x; fused "both" reads
            // the values the row pass stored; fused "col" evaluates the op here
            constexpr bool kEval = (MODE == kCol) && (OP != kQuant);
            constexpr int kSrc = (MODE == kBoth) ? (NIN - NOUT) : 0;
            const uint32_t crow = kSub * srb + static_cast<uint32_t>(lane);
            const uint32_t cc = static_cast<uint32_t>(lane >> 2);   // column within a unit
            // stmatrix row address of this lane (lanes 0-15): matrix t/8 = which
            // 16-byte half of column (t%8)'s 32 staged bytes, halves swapped for
            // columns with bit 2 set (conflict-free for both the stores and the
            // reads below)
            const uint32_t t16 = static_cast<uint32_t>(lane) & 15u;
            const uint32_t stg_row = smem_u32(stg) + (t16 & 7u) * 32u + (((t16 >> 3) ^ ((t16 >> 2) & 1u)) * 16u);
            const int64_t left64 = a.N - (c0 + cc);
            const int cols_left = left64 > 32 ? 32 : static_cast<int>(left64 < 0 ? 0 : left64);
            const bool row_ok = r0 < a.M;
            uint8_t *sp[2];
#pragma unroll
            for (int o = 0; o < NOUT; ++o) sp[o] = a.s_col[o] + (r0 >> 5) * a.ld_scol + (c0 + cc);
#pragma unroll kUnroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t off = swz(crow, chunk0 + k);
                uint32_t out[2][4];
                uint32_t amax[2];
                const bool live = row_ok && (8 * k < cols_left);
                if constexpr (kEval) {
                    uint32_t in[3][4];
                    uint64_t hv[2][4];
#pragma unroll
                    for (int i = 0; i < NIN; ++i) ldsm_x4_trans(stage + i * kTileBytes + off, in[i]);
                    const uint32_t near = elements8<OP, true>(in, out, hv);
#pragma unroll
                    for (int o = 0; o < NOUT; ++o) amax[o] = amax32_lanes4(out[o]);
                    settle<OP, true>(a, in, out, amax, near, hv);
                } else {
#pragma unroll
                    for (int o = 0; o < NOUT; ++o) {
                        ldsm_x4_trans(stage + (kSrc + o) * kTileBytes + off, out[o]);
                        amax[o] = amax32_lanes4(out[o]);
                    }
                }
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    uint32_t w0, w1;
                    const uint32_t sc = encode_block8(out[o], amax[o], w0, w1);
                    // w0 = codes of rows 2q, 2q+1, 8+2q, 9+2q of column 8k + cc,
                    // w1 the same 16 rows further; they land at bytes 4q..4q+3
                    // of the column's two 16-byte halves (row order restored
                    // when the column is read back)
                    stsm_x2(stg_row + static_cast<uint32_t>(o * 1024 + k * 256), w0, w1);
                    if (live && q == 0) sp[o][8 * k] = static_cast<uint8_t>(sc);
                }
            }
            __syncwarp();
            // each lane stores one column's 32 codes
            const int64_t gcol = c0 + lane;
            if (r0 < a.M && gcol < a.N) {
                int64_t grp = 0, rin = r0;
                if (a.group_stride != 0) {  // 3D: per-expert column-major output
                    grp = r0 / a.group_rows;
                    rin = r0 - grp * a.group_rows;
                }
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    const uint8_t *src = stg + o * 1024 + lane * 32;
                    const uint32_t sw = ((static_cast<uint32_t>(lane) >> 2) & 1u) * 16u;
                    const uint4 lo = *reinterpret_cast<const uint4 *>(src + (0u ^ sw));
                    const uint4 hi = *reinterpret_cast<const uint4 *>(src + (16u ^ sw));
                    // staged words hold rows (j, j+1, j+8, j+9), j = 0, 2, 4, 6
                    const uint4 r_lo = make_uint4(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410),
                                                  __byte_perm(lo.x, lo.y, 0x7632), __byte_perm(lo.z, lo.w, 0x7632));
                    const uint4 r_hi = make_uint4(__byte_perm(hi.x, hi.y, 0x5410), __byte_perm(hi.z, hi.w, 0x5410),
                                                  __byte_perm(hi.x, hi.y, 0x7632), __byte_perm(hi.z, hi.w, 0x7632));
                    uint4 *dst = reinterpret_cast<uint4 *>(a.q_col[o] + grp * a.group_stride +
                                                           gcol * a.ld_qcol + rin);
                    __stcs(dst, r_lo);
                    __stcs(dst + 1, r_hi);
                }
            }
            __syncwarp();
        }

        if constexpr (kSplit) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
}

}  // namespace mx
