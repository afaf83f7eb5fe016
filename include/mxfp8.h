/*
 * mxfp8.h -- C ABI of libmxfp8: MXFP8 casts for MoE training on GB300 (sm_103a).
 *
 * MXFP8 here means: E4M3 (fn) data plus one E8M0 scale byte per block of 32
 * consecutive elements along the blocking axis.  The scale byte is RCEIL:
 * e = ceil(log2(amax / 448)) clamped to [-127, 127], byte = e + 127, and 0
 * for an all-zero block; a block whose amax is NaN or Inf gets byte 255 and
 * 32 NaN codes (0x7F).  Data codes are x * 2^-e rounded to nearest, ties to
 * even, saturating at +-448, sign of zero kept (a byte-0 scale multiplies by
 * 2^127).  Sources: "Add swiglu + MXFP8 fused CuTe DSL kernel" (torchao fork
 * PR #2), sections "Summary", "API" and "Numerics and tests" and its commit
 * message; "[mxfp8 moe training] update 3d quant colwise scaling kernel to use
 * single input/output TMA descriptors" (pytorch/ao PR #3034), "Summary".
 *
 * Conventions shared by every entry point:
 *  - bf16 tensors are passed as pointers to their 16-bit patterns.
 *  - All tensor pointers are DEVICE pointers on the current CUDA device; the
 *    caller owns every buffer.  The library never allocates a buffer for a
 *    call, never frees one and never synchronizes; work is enqueued on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - Sizes and leading dimensions are int64_t, in ELEMENTS (bf16 elements for
 *    inputs, bytes for E4M3/E8M0 outputs).  Indexing is 64-bit.
 *  - Rowwise (1x32 blocks along a row): data (M, N) row-major, element (r, c)
 *    at q_row[r * ld_qrow + c]; scales (M, N/32) row-major, s_row[r * ld_srow
 *    + c/32].  Needs N % 32 == 0.
 *  - Colwise (32x1 blocks down a column): data (M, N) COLUMN-major, element
 *    (r, c) at q_col[c * ld_qcol + r]; scales (M/32, N) row-major,
 *    s_col[(r/32) * ld_scol + c].  Needs M % 32 == 0.
 *  - Pointers of a disabled direction are ignored (pass NULL).
 *  - M == 0 or N == 0 (or E == 0) is an empty call: MXFP8_OK, nothing runs.
 *  - Errors are returned, never thrown; every argument check runs on the host
 *    before anything is enqueued, so a rejected call leaves the stream and
 *    the device untouched.
 *  - Alignment: input pointers 16-byte aligned and ld * 2 a multiple of 16
 *    bytes (TMA tiles); E4M3 data pointers 16-byte aligned with leading
 *    dimensions multiples of 16.  Scale pointers have no alignment rule.
 *  - No output may overlap an input or another output (strided regions with
 *    equal leading dimensions are checked exactly, so interleaved layouts
 *    such as [dGate | dUp] halves of one buffer are accepted).
 *  - Calls are thread-safe.  The first call on a device builds 2 MB of
 *    read-only tables in device memory (see mxfp8_init); do that before
 *    capturing a CUDA graph.
 */
#ifndef MXFP8_H
#define MXFP8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP8_ROWWISE = 1, /* 1x32 blocks, row-major data + (M, N/32) scales     */
    MXFP8_COLWISE = 2, /* 32x1 blocks, column-major data + (M/32, N) scales  */
    MXFP8_BOTH = 3,    /* both sets from one read of the input               */
    /*
     * Flag, OR-ed into any of the three (2D quantizer and the SwiGLU entry
     * points): scales come out in the blocked layout that block-scaled
     * tensor-core GEMMs read ("the same blocked tcgen05 layouts as the
     * standalone quantizers", "Add swiglu + MXFP8 fused CuTe DSL kernel",
     * commit message; 128 x 4 tiles, "[mxfp8 moe training] add compile
     * support", review thread).  The row scales, as the (M, N/32) matrix, and
     * the column scales, as the (N, M/32) matrix (column c's blocks along
     * its rows), are padded to R' = 128 ceil(R/128) rows and C' = 4
     * ceil(C/4) columns and cut into 128 x 4 tiles stored one after another
     * row-major, 512 bytes each; entry (r, c) of a tile sits at byte
     * (r % 32) * 16 + (r / 32) * 4 + c.  Each scale buffer then holds R' * C'
     * bytes and its leading dimension is ignored; row-scale buffers must be
     * 4-byte aligned.  Padding entries are left as they were or set to 0:
     * pass zero-filled buffers.
     */
    MXFP8_BLOCKED_SCALES = 8
} mxfp8_scale_mode;

typedef enum {
    MXFP8_OK = 0,
    MXFP8_ERR_NULL = 1,     /* a required pointer is NULL                        */
    MXFP8_ERR_SHAPE = 2,    /* negative size, or N % 32 (rowwise) / M % 32
                               (colwise, 3D N) not zero, or a size overflows
                               (M or N above 2^31 - 256, more than about 2^31
                               tiles of 96 x 128, a byte extent past int64)      */
    MXFP8_ERR_ALIGN = 3,    /* pointer or leading dimension misaligned           */
    MXFP8_ERR_LD = 4,       /* leading dimension smaller than the row it spans   */
    MXFP8_ERR_MODE = 5,     /* scale mode not 1, 2 or 3                          */
    MXFP8_ERR_OVERLAP = 6,  /* an output overlaps an input or another output     */
    MXFP8_ERR_LAUNCH = 7,   /* the CUDA runtime refused the launch               */
    MXFP8_ERR_DEVICE = 8,   /* no usable device, or device set-up failed         */
    MXFP8_ERR_CAPTURE = 9   /* first call on a device made during stream capture */
} mxfp8_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *mxfp8_status_str(mxfp8_status s);

/* Version of this library: major * 10000 + minor * 100 + patch. */
int mxfp8_version(void);

/*
 * One-time set-up of the current device: fills the library's read-only
 * tables -- one entry per bf16 pattern g of sigmoid(g) in double and as a
 * (hi, lo) float pair, and of Phi(g) and gelu'(g) as (hi, lo) pairs and in
 * double (used by the exact-rounding paths of the SwiGLU and GEGLU
 * kernels), and the GEGLU fast path's table of (Phi(-t), t phi(t)) over
 * the bf16 magnitudes t from 2^-20 to 6 (3 MB in all) -- and waits for them
 * on `stream`.  Every entry point calls it
 * on its first use on a device; call it yourself before capturing a graph.
 * Returns MXFP8_ERR_CAPTURE if it would have to run inside a capture.
 */
mxfp8_status mxfp8_init(void *stream);

/*
 * Standalone 2D quantizer: bf16 x (M, N), element (r, c) at x[r * ld_x + c],
 * to MXFP8 rowwise, colwise or both, in one pass over x.
 * ("Add swiglu + MXFP8 fused CuTe DSL kernel", sections "Summary" and
 * "Numerics and tests": the standalone MXFP8 quantizers.)
 */
mxfp8_status mxfp8_quant_2d(const uint16_t *x, int64_t ld_x, int64_t M, int64_t N,
                            int mode,
                            uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                            uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                            void *stream);

/*
 * Fused SwiGLU forward + MXFP8 cast.  h = silu(gate) * up, evaluated at fp32
 * precision and rounded once to bf16 (never written to memory), is cast as
 * mxfp8_quant_2d would cast a stored h.  gate and up are (M, N) with the same
 * leading dimension ld_in; the packed [gate | up] buffer of a fused w13
 * projection is gate = buf, up = buf + N, ld_in = 2N.
 * ("Add swiglu + MXFP8 fused CuTe DSL kernel", sections "Summary" and "API".)
 */
mxfp8_status mxfp8_swiglu_fwd(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                              int64_t M, int64_t N, int mode,
                              uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                              uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                              void *stream);

/*
 * The fused forward that also writes the bf16 activation h (M, N) row-major
 * at h[r * ld_h + c], for recipes whose weight-gradient GEMMs take h in bf16
 * ("Add swiglu + MXFP8 fused CuTe DSL kernel", section "Summary": the
 * BF16-wgrad recipe, where the kernel emits rowwise-only casts and the
 * activation is otherwise recomputed in bf16 at the autograd boundary).  The
 * h written is the value the cast encoded: within one bf16 step of the
 * correctly rounded activation (equal to it for all but about 1e-4 of the
 * elements; see mxfp8_swiglu_fwd).  Needs the rowwise direction in `mode`
 * (MXFP8_ERR_MODE otherwise); h non-NULL, 16-byte aligned, ld_h >= N with
 * ld_h * 2 a multiple of 16; h may not overlap any other argument.  Every
 * other argument as in mxfp8_swiglu_fwd.
 */
mxfp8_status mxfp8_swiglu_fwd_with_h(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                                     int64_t M, int64_t N, int mode, uint16_t *h, int64_t ld_h,
                                     uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                                     uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                                     void *stream);

/*
 * Fused SwiGLU backward + MXFP8 cast.  From dh (M, N), gate and up:
 *   dgate = dh * up * sigmoid(gate) * (1 + gate * (1 - sigmoid(gate)))
 *   dup   = dh * gate * sigmoid(gate)
 * each evaluated at fp32 precision, rounded once to bf16, then cast like
 * mxfp8_quant_2d.  dgate and dup share the leading dimensions of their
 * direction, so the concatenated [dGate | dUp] outputs are: rowwise
 * du_row = dg_row + N with ld_qrow = 2N (scales du_srow = dg_srow + N/32,
 * ld_srow = N/16); colwise du_col = dg_col + N * ld_qcol and
 * du_scol = dg_scol + N with ld_scol = 2N.
 * ("Add swiglu + MXFP8 fused CuTe DSL kernel", sections "API" and "Numerics
 * and tests".)
 */
mxfp8_status mxfp8_swiglu_bwd(const uint16_t *dh, int64_t ld_dh,
                              const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                              int64_t M, int64_t N, int mode,
                              uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow,
                              uint8_t *dg_srow, uint8_t *du_srow, int64_t ld_srow,
                              uint8_t *dg_col, uint8_t *du_col, int64_t ld_qcol,
                              uint8_t *dg_scol, uint8_t *du_scol, int64_t ld_scol,
                              void *stream);

/*
 * Per-expert 3D colwise quantizer: x (E, N, K) bf16 row-major (element
 * (e, n, k) at x[(e*N + n)*K + k]) -> E4M3 data column-major per expert,
 * element (e, n, k) at q[e*N*K + k*N + n], and E8M0 scales (E, N/32, K)
 * row-major, s[e*(N/32)*K + (n/32)*K + k]; blocks of 32 along N.  One launch
 * covers every expert.  Needs N % 32 == 0 and K % 8 == 0.
 * ("[mxfp8 moe training] update 3d quant colwise scaling kernel to use
 * single input/output TMA descriptors", sections "Summary" and "Performance".)
 */
mxfp8_status mxfp8_quant_3d_colwise(const uint16_t *x, int64_t E, int64_t N, int64_t K,
                                    uint8_t *q, uint8_t *s, void *stream);

/*
 * Per-expert 3D quantizer, either or both directions from one read of x
 * (E, N, K) bf16 row-major:
 *  - rowwise (1x32 blocks along K): data (E, N, K) row-major, q_row[(e*N +
 *    n)*K + k]; scales (E, N, K/32) row-major.  Needs K % 32 == 0.
 *  - colwise (32x1 blocks along N): the layout of mxfp8_quant_3d_colwise.
 *    Needs N % 32 == 0.
 * With MXFP8_BLOCKED_SCALES each expert's scale matrix -- rowwise (N, K/32),
 * colwise (K, N/32) (column k's blocks along its row) -- is laid out as in
 * that flag's description, the experts one after another: E * R' * C' bytes
 * per buffer (R', C' the padded rows and columns of one expert's matrix);
 * needs N % 32 == 0 ("[mxfp8 moe training] add compile support": the
 * per-group 3D scale swizzle, the 3D cast the perf analysis asks for).
 * K % 8 == 0 always.
 */
mxfp8_status mxfp8_quant_3d(const uint16_t *x, int64_t E, int64_t N, int64_t K, int mode,
                            uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                            void *stream);

/*
 * Per-group blocked scales for grouped-GEMM operands ("[mxfp8 moe training]
 * add compile support": the M-groups and K-groups scale swizzles, padded
 * rows + 128 * groups and cols + 4 * groups): the M rows of the input form
 * G consecutive token groups, group_end[g] (device memory, int32) the end
 * row of group g (cumulative; non-decreasing; every end but the last a
 * multiple of 32; the last = M; 1 <= G <= 256).  The data outputs are those
 * of the ungrouped calls; the scales always come out blocked (see
 * MXFP8_BLOCKED_SCALES, which `mode` may carry or not):
 *  - row scales (M-groups): group g's rows of the (M, N/32) matrix start on
 *    a fresh 128-row tile, at the sum of the earlier groups' sizes rounded
 *    up to 128; the buffer holds (ceil(M/128) + G) * 128 rows of
 *    4 * ceil(N/128) bytes;
 *  - column scales (K-groups): group g's columns of the (N, M/32) matrix
 *    start on a fresh 4-column tile, at the sum of the earlier groups'
 *    block counts rounded up to 4; the matrix has (ceil(M/128) + G) * 4
 *    columns and 128 * ceil(N/128) rows.
 * Entries outside the groups are not written: pass zero-filled buffers.
 * The group ends are checked on the device (they are never read by the
 * host, so the call does not synchronise): if they break a rule, no scale
 * is written and status bit 4 is set (mxfp8_device_status).  Other
 * arguments and errors as in mxfp8_quant_2d / mxfp8_swiglu_fwd /
 * mxfp8_swiglu_bwd; `act` selects the gated activation (0 SwiGLU, 1 GEGLU;
 * else MXFP8_ERR_MODE).
 */
mxfp8_status mxfp8_quant_2d_grouped(const uint16_t *x, int64_t ld_x, int64_t M, int64_t N, int mode,
                                    const int32_t *group_end, int64_t num_groups,
                                    uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                                    uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, void *stream);
mxfp8_status mxfp8_swiglu_fwd_grouped(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                                      int64_t M, int64_t N, int mode, int act,
                                      const int32_t *group_end, int64_t num_groups,
                                      uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                                      uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, void *stream);
mxfp8_status mxfp8_swiglu_bwd_grouped(const uint16_t *dh, int64_t ld_dh,
                                      const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                                      int64_t M, int64_t N, int mode, int act,
                                      const int32_t *group_end, int64_t num_groups,
                                      uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow,
                                      uint8_t *dg_srow, uint8_t *du_srow,
                                      uint8_t *dg_col, uint8_t *du_col, int64_t ld_qcol,
                                      uint8_t *dg_scol, uint8_t *du_scol, void *stream);

/*
 * Allocation-free forward, for callers that cannot call cudaMalloc at all:
 * code that must live inside a host framework's fixed device-memory arena,
 * or that runs where allocation is forbidden.  (The pages have no
 * counterpart: this is the unfused order -- activation, then the standalone
 * cast -- with the activation kept in library-owned scratch.)
 * Same arguments and rules as mxfp8_swiglu_fwd: pass 1 writes the bf16
 * activation h, every element correctly rounded (the fused kernel's exact
 * path), into a static scratch array; pass 2 casts h with the standalone
 * quantizer.  Results: scale bytes equal the fused forward's; data codes are
 * the plain definition's bit for bit, where the fused forward's may differ
 * by one code in rare elements (its fast activation is within one bf16 step
 * of the exact one).
 *  - Scratch: 8,388,608 bf16 elements (16 MiB) reserved in every device that
 *    loads the library, held until the process exits.  Rows are padded to a
 *    multiple of 8 elements, so the limit is M * roundup(N, 8) <= 8,388,608;
 *    larger problems return MXFP8_ERR_SHAPE before anything is enqueued.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *  - The first call on a device looks up the scratch's device address (and
 *    does the library's one-time set-up, see mxfp8_init); make that first
 *    call before any stream capture.
 *  - Every call shares the one scratch array and overwrites the part it uses
 *    before reading it; calls that overlap on the GPU (on different streams)
 *    race on it and must be ordered by the caller.
 */
mxfp8_status mxfp8_swiglu_fwd_noalloc(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                                      int64_t M, int64_t N, int mode,
                                      uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                                      uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                                      void *stream);

/*
 * GEGLU: the same fused forward and backward with the activation gelu(g) =
 * g * Phi(g), Phi the standard normal CDF (exact erf form), in place of
 * silu ("Add swiglu + MXFP8 fused CuTe DSL kernel", section "API": the
 * activation is a compile-time policy of the one kernel).  h = gelu(gate) *
 * up; dgate = dh * up * (Phi(gate) + gate * phi(gate)) with phi the normal
 * density, dup = dh * gelu(gate).  Arguments, layouts, rules, errors and the
 * tolerance are those of mxfp8_swiglu_fwd / mxfp8_swiglu_bwd.
 */
mxfp8_status mxfp8_geglu_fwd(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                             int64_t M, int64_t N, int mode,
                             uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                             uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                             void *stream);
mxfp8_status mxfp8_geglu_bwd(const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                             const uint16_t *up, int64_t ld_in, int64_t M, int64_t N, int mode,
                             uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow,
                             uint8_t *dg_srow, uint8_t *du_srow, int64_t ld_srow,
                             uint8_t *dg_col, uint8_t *du_col, int64_t ld_qcol,
                             uint8_t *dg_scol, uint8_t *du_scol, int64_t ld_scol, void *stream);

/*
 * Sticky device-side status of the current device.  Kernels never trap: a
 * pipeline wait that exceeds its limit (about a second) makes the kernel set
 * a flag bit and return.  flags: bit 0 consumer wait, bit 1 producer wait,
 * bit 2 drain wait, bit 3 self-test wait, bit 4 invalid group ends.
 * fallbacks: number of SwiGLU or GEGLU elements the fused kernels sent
 * through their rare path (both elements of every pair settled there: pairs
 * holding a value near a scale boundary, a gate outside the fast range or a
 * non-finite value, and every pair of a block with a huge amax); the rare
 * path recomputes exactly the elements among them that need it.
 * Synchronizes `stream`; with reset != 0 clears both afterwards.
 * Either output pointer (host memory) may be NULL.
 */
mxfp8_status mxfp8_device_status(uint32_t *flags, uint64_t *fallbacks, int reset, void *stream);

/*
 * Self-test of the SwiGLU fast path: writes, for every bf16 bit pattern g
 * (index g), the fp32 factors the kernels compute -- out[k*65536 + g] for
 * k = 0 sigmoid(g), 1 2^60 silu(g) (the forward's scaled form), 2 1 -
 * sigmoid(g), 3 1 + g(1 - sigmoid(g)), 4 silu'(g), 5 2^120 e^g (the factor of
 * the wide-range values the kernels use for gates below -16).  `out` is a
 * device buffer of 6 * 65536 floats, 16-byte aligned.  The tests compare these with the
 * exact factors: the error bounds they establish are the ones the fused
 * kernels' recomputation windows are sized for.
 */
mxfp8_status mxfp8_selftest_activation(float *out, void *stream);

/*
 * Self-test of the GEGLU fast paths, like mxfp8_selftest_activation: for
 * every bf16 pattern g, out[k*65536 + g] for k = 0 Phi(g), 1 gelu(g), 2
 * gelu'(g) = Phi(g) + g phi(g) from the tail table (the forward, and the
 * backward's "both" mode with per-group scales), 3 Phi(g) and 4 gelu'(g)
 * from the rational tail (the rest of the backward).  `out` is a device buffer of
 * 5 * 65536 floats, 16-byte aligned.
 */
mxfp8_status mxfp8_selftest_activation_gelu(float *out, void *stream);

/*
 * Failure-detection self-test: launches one thread that waits on a shared
 * memory barrier nobody arrives on, giving up after `limit_cycles` SM clock
 * cycles; it then sets status bit 3 and returns.  Used by the tests to show
 * that a stuck wait ends with a readable error instead of a hang.
 */
mxfp8_status mxfp8_selftest_wait_timeout(uint64_t limit_cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_H */
