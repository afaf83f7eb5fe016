// kernel.cuh -- the persistent tile kernel shared by every entry point.
//
// One CTA per SM.  Warp 8 is the producer: its lane 0 streams the input tiles
// (128 rows x 64 bf16 columns per tensor, 128-byte swizzle) into a ring of
// shared-memory stages with TMA, each stage guarded by a "full" mbarrier
// (transaction bytes) and an "empty" mbarrier (one arrive per consumer warp).
// Warps 0..7 are consumers; per tile they
//   row pass  : each thread owns one 1x32 block (row 16w + lane/2, block
//               lane%2), evaluates the element op from four 16-byte shared
//               loads per input and encodes the rowwise MXFP8 block;
//   col pass  : warp w owns the 8-column chunk w; ldmatrix.trans hands each
//               group of four lanes one column of a 32-row block, which is
//               encoded colwise and written as 8-byte pieces of the
//               column-major output.
// In "both" mode the row pass writes the bf16 element values back into the
// stage (over an input it no longer needs) and a named barrier separates the
// passes, so both scale sets come from one read of the inputs.  In "col" mode
// the element op runs directly on the transposed fragments.
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

template <int OP>
constexpr int default_stages()
{
    return OP == kQuant ? 8 : (OP == kFwd ? 4 : 3);
}

template <int OP, int STAGES>
constexpr size_t smem_bytes()
{
    return 1024 + static_cast<size_t>(STAGES) * OpTraits<OP>::kIn * kTileBytes + 2 * STAGES * 8;
}

// ------------------------------------------------------------- row pass op
// Evaluate the element op for one thread's 32 elements (16 packed words per
// input) into out[o][16].
template <int OP>
__device__ __forceinline__ void row_elements(const KernelArgs &a, const uint32_t (&in)[3][16],
                                             uint32_t (&out)[2][16])
{
    if constexpr (OP == kQuant) {
#pragma unroll
        for (int i = 0; i < 16; ++i) out[0][i] = in[0][i];
    } else if constexpr (OP == kFwd) {
        uint32_t bad = 0;
        float hv[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float g0 = bf16lo(in[0][i]), g1 = bf16hi(in[0][i]);
            const float u0 = bf16lo(in[1][i]), u1 = bf16hi(in[1][i]);
            const bool ok0 = swiglu_h_fast(g0, u0, hv[2 * i]);
            const bool ok1 = swiglu_h_fast(g1, u1, hv[2 * i + 1]);
            bad |= (ok0 ? 0u : 1u) << (2 * i);
            bad |= (ok1 ? 0u : 1u) << (2 * i + 1);
        }
        if (bad) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (bad & (1u << e)) {
                    const uint32_t gw = in[0][e >> 1], uw = in[1][e >> 1];
                    const float g = (e & 1) ? bf16hi(gw) : bf16lo(gw);
                    const float u = (e & 1) ? bf16hi(uw) : bf16lo(uw);
                    hv[e] = swiglu_h_exact(a.sig_table, g, u);
                }
            }
        }
        count_fallbacks(a.fallbacks, bad);
#pragma unroll
        for (int i = 0; i < 16; ++i) out[0][i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
    } else {
        uint32_t bad_g = 0, bad_u = 0;
        float dg[32], du[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int e = 2 * i + k;
                const float d = k ? bf16hi(in[0][i]) : bf16lo(in[0][i]);
                const float g = k ? bf16hi(in[1][i]) : bf16lo(in[1][i]);
                const float u = k ? bf16hi(in[2][i]) : bf16lo(in[2][i]);
                const uint32_t m = swiglu_grads_fast(d, g, u, dg[e], du[e]);
                bad_g |= (m & 1u) << e;
                bad_u |= ((m >> 1) & 1u) << e;
            }
        }
        const uint32_t bad = bad_g | bad_u;
        if (bad) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (bad & (1u << e)) {
                    const int i = e >> 1, k = e & 1;
                    const float d = k ? bf16hi(in[0][i]) : bf16lo(in[0][i]);
                    const float g = k ? bf16hi(in[1][i]) : bf16lo(in[1][i]);
                    const float u = k ? bf16hi(in[2][i]) : bf16lo(in[2][i]);
                    float xg, xu;
                    swiglu_grads_exact(a.sig_table, d, g, u, xg, xu);
                    if (bad_g & (1u << e)) dg[e] = xg;
                    if (bad_u & (1u << e)) du[e] = xu;
                }
            }
        }
        count_fallbacks(a.fallbacks, bad_g);
        count_fallbacks(a.fallbacks, bad_u);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            out[0][i] = pack_bf16x2(dg[2 * i], dg[2 * i + 1]);
            out[1][i] = pack_bf16x2(du[2 * i], du[2 * i + 1]);
        }
    }
}

// Same op on a transposed fragment: 4 packed words (8 elements) per input.
template <int OP>
__device__ __forceinline__ void col_elements(const KernelArgs &a, const uint32_t (&in)[3][4],
                                             uint32_t (&out)[2][4])
{
    if constexpr (OP == kQuant) {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[0][i] = in[0][i];
    } else if constexpr (OP == kFwd) {
        uint32_t bad = 0;
        float hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok0 = swiglu_h_fast(bf16lo(in[0][i]), bf16lo(in[1][i]), hv[2 * i]);
            const bool ok1 = swiglu_h_fast(bf16hi(in[0][i]), bf16hi(in[1][i]), hv[2 * i + 1]);
            bad |= (ok0 ? 0u : 1u) << (2 * i);
            bad |= (ok1 ? 0u : 1u) << (2 * i + 1);
        }
        if (bad) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (bad & (1u << e)) {
                    const uint32_t gw = in[0][e >> 1], uw = in[1][e >> 1];
                    const float g = (e & 1) ? bf16hi(gw) : bf16lo(gw);
                    const float u = (e & 1) ? bf16hi(uw) : bf16lo(uw);
                    hv[e] = swiglu_h_exact(a.sig_table, g, u);
                }
            }
        }
        count_fallbacks(a.fallbacks, bad);
#pragma unroll
        for (int i = 0; i < 4; ++i) out[0][i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
    } else {
        uint32_t bad_g = 0, bad_u = 0;
        float dg[8], du[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = e >> 1, k = e & 1;
            const float d = k ? bf16hi(in[0][i]) : bf16lo(in[0][i]);
            const float g = k ? bf16hi(in[1][i]) : bf16lo(in[1][i]);
            const float u = k ? bf16hi(in[2][i]) : bf16lo(in[2][i]);
            const uint32_t m = swiglu_grads_fast(d, g, u, dg[e], du[e]);
            bad_g |= (m & 1u) << e;
            bad_u |= ((m >> 1) & 1u) << e;
        }
        const uint32_t bad = bad_g | bad_u;
        if (bad) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (bad & (1u << e)) {
                    const int i = e >> 1, k = e & 1;
                    const float d = k ? bf16hi(in[0][i]) : bf16lo(in[0][i]);
                    const float g = k ? bf16hi(in[1][i]) : bf16lo(in[1][i]);
                    const float u = k ? bf16hi(in[2][i]) : bf16lo(in[2][i]);
                    float xg, xu;
                    swiglu_grads_exact(a.sig_table, d, g, u, xg, xu);
                    if (bad_g & (1u << e)) dg[e] = xg;
                    if (bad_u & (1u << e)) du[e] = xu;
                }
            }
        }
        count_fallbacks(a.fallbacks, bad_g);
        count_fallbacks(a.fallbacks, bad_u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[0][i] = pack_bf16x2(dg[2 * i], dg[2 * i + 1]);
            out[1][i] = pack_bf16x2(du[2 * i], du[2 * i + 1]);
        }
    }
}

// ------------------------------------------------------------------ stores
__device__ __forceinline__ void store_row_block(const KernelArgs &a, int o, int64_t row,
                                                int64_t col, const uint32_t (&codes)[8],
                                                uint32_t scale)
{
    uint8_t *q = a.q_row[o] + row * a.ld_qrow + col;
    uint4 *q4 = reinterpret_cast<uint4 *>(q);
    __stcs(q4, make_uint4(codes[0], codes[1], codes[2], codes[3]));
    __stcs(q4 + 1, make_uint4(codes[4], codes[5], codes[6], codes[7]));
    a.s_row[o][row * a.ld_srow + (col >> 5)] = static_cast<uint8_t>(scale);
}

// colwise piece: rows row0 + 8q .. +7 of column col (row0 a multiple of 32)
__device__ __forceinline__ void store_col_piece(const KernelArgs &a, int o, int64_t row0,
                                                int64_t col, uint32_t q, uint32_t w0, uint32_t w1,
                                                uint32_t scale)
{
    const int64_t grp = row0 / a.group_rows;
    const int64_t rin = row0 - grp * a.group_rows;
    uint8_t *dst = a.q_col[o] + grp * a.group_stride + col * a.ld_qcol + rin + 8 * q;
    __stcs(reinterpret_cast<uint2 *>(dst), make_uint2(w0, w1));
    if (q == 0) a.s_col[o][(row0 >> 5) * a.ld_scol + col] = static_cast<uint8_t>(scale);
}

// ------------------------------------------------------------------ kernel
template <int OP, int MODE, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp8_tile_kernel(const __grid_constant__ CUtensorMap tm0,
                      const __grid_constant__ CUtensorMap tm1,
                      const __grid_constant__ CUtensorMap tm2, const KernelArgs a)
{
    constexpr int NIN = OpTraits<OP>::kIn;
    constexpr int NOUT = OpTraits<OP>::kOut;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * NIN * kTileBytes);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    const int64_t num_tiles = a.num_tiles;
    const int64_t tiles_n = a.tiles_n;

    // ------------------------------------------------------- producer warp
    if (warp == kConsumerWarps) {
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
                if (NIN > 1) tma_load_2d(dst + kTileBytes, &tm1, c0, r0, bar);
                if (NIN > 2) tma_load_2d(dst + 2 * kTileBytes, &tm2, c0, r0, bar);
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
    const uint32_t rrow = static_cast<uint32_t>(16 * warp + (lane >> 1));  // row-pass row
    const uint32_t rblk = static_cast<uint32_t>(lane & 1);                  // row-pass block
    const uint32_t q = static_cast<uint32_t>(lane & 3);
    const uint32_t ccol = static_cast<uint32_t>(8 * warp + (lane >> 2));    // col-pass column

    // the fused "both" mode hands values from the row pass to the col pass
    // through shared memory, separated by a named barrier
    constexpr bool kSync = (MODE == kBoth) && (OP != kQuant);
    int it = 0;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = static_cast<uint32_t>(it / STAGES) & 1u;
        bool fail = !mbar_wait_bounded(full0 + 8 * s, ph, a.wait_limit);
        fail = __any_sync(0xFFFFFFFFu, fail);
        if (fail && !kSync) {
            if (lane == 0) atomicOr(a.status, kStatusConsumerWait);
            return;
        }
        const int64_t r0 = (t / tiles_n) * kTileM;
        const int64_t c0 = (t % tiles_n) * kTileN;
        const uint32_t stage = smem_base + static_cast<uint32_t>(s * NIN) * kTileBytes;
        uint8_t *stage_ptr = smem + static_cast<size_t>(s * NIN) * kTileBytes;

        if constexpr (MODE & kRow) {
            if (!fail) {
                uint32_t in[3][16];
                uint32_t out[2][16];
#pragma unroll
                for (int i = 0; i < NIN; ++i) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            stage_ptr + i * kTileBytes + swz(rrow, 4 * rblk + k));
                        in[i][4 * k + 0] = v.x;
                        in[i][4 * k + 1] = v.y;
                        in[i][4 * k + 2] = v.z;
                        in[i][4 * k + 3] = v.w;
                    }
                }
                row_elements<OP>(a, in, out);
                const int64_t grow = r0 + rrow;
                const int64_t gcol = c0 + 32 * rblk;
                const bool live = (grow < a.M) && (gcol < a.N);
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    uint32_t codes[8];
                    const uint32_t sc = encode_block32(out[o], codes);
                    if (live) store_row_block(a, o, grow, gcol, codes, sc);
                }
                if constexpr (kSync) {
                    // element values back into the stage for the col pass:
                    // output o overwrites input (NIN - NOUT + o)
#pragma unroll
                    for (int o = 0; o < NOUT; ++o) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            *reinterpret_cast<uint4 *>(stage_ptr + (NIN - NOUT + o) * kTileBytes +
                                                       swz(rrow, 4 * rblk + k)) =
                                make_uint4(out[o][4 * k], out[o][4 * k + 1], out[o][4 * k + 2],
                                           out[o][4 * k + 3]);
                        }
                    }
                }
            }
        }

        if constexpr (kSync) {
            fail = consumers_sync_or(fail);
            if (fail) {
                if (tid == 0) atomicOr(a.status, kStatusConsumerWait);
                return;
            }
        }

        if constexpr (MODE & kCol) {
            // element values for the col pass: quant reads x; fused "both" reads
            // the values the row pass stored; fused "col" evaluates the op here
            constexpr bool kEval = (MODE == kCol) && (OP != kQuant);
            constexpr int kSrc = (MODE == kBoth) ? (NIN - NOUT) : 0;
            const int64_t gcol = c0 + ccol;
#pragma unroll
            for (int rb = 0; rb < kTileM / 32; ++rb) {
                const uint32_t lrow = static_cast<uint32_t>(32 * rb + lane);
                const uint32_t off = swz(lrow, static_cast<uint32_t>(warp));
                uint32_t out[2][4];
                if constexpr (kEval) {
                    uint32_t in[3][4];
#pragma unroll
                    for (int i = 0; i < NIN; ++i) ldsm_x4_trans(stage + i * kTileBytes + off, in[i]);
                    col_elements<OP>(a, in, out);
                } else {
#pragma unroll
                    for (int o = 0; o < NOUT; ++o)
                        ldsm_x4_trans(stage + (kSrc + o) * kTileBytes + off, out[o]);
                }
                const int64_t row0 = r0 + 32 * rb;
                const bool live = (row0 < a.M) && (gcol < a.N);
#pragma unroll
                for (int o = 0; o < NOUT; ++o) {
                    uint32_t w0, w1;
                    const uint32_t sc = encode_col32(out[o], q, w0, w1);
                    if (live) store_col_piece(a, o, row0, gcol, q, w0, w1, sc);
                }
            }
        }

        if constexpr (kSync) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
}

}  // namespace mx
