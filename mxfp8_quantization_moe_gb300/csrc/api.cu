// api.cu -- the C ABI of libmxfp8 (declared in include/mxfp8.h): argument
// validation on the host, TMA descriptor encoding, per-device set-up, launch.
//
// Every argument check runs before anything touches the CUDA runtime, so a
// rejected call returns a status code without side effects (and can be made
// on a machine without a GPU).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.cuh"
#include "mxfp8.h"

namespace {

using mx::KernelArgs;

// ----------------------------------------------------- device-side state
// Read-only tables, one entry per bf16 bit pattern g (sigmoid(g) in double
// and as a (hi, lo) float pair; (hi, lo) pairs of Phi(g) and gelu'(g), and
// the two in double),
// sticky status bits and the count of elements settled by the exact path.
// Each device that loads the library holds its own copy.
__device__ double g_sig_table[65536];
__device__ float2 g_sig2_table[65536];
__device__ float4 g_gelu_table[65536];
__device__ double2 g_gelu_dtable[65536];
__device__ float2 g_gelu_tail[mx::kGeluTabN];
__device__ unsigned g_status;
__device__ unsigned long long g_fallbacks;

__device__ __forceinline__ float2 float_pair(double v)
{
    const float hi = __double2float_rn(v);
    return make_float2(hi, __double2float_rn(__dadd_rn(v, -static_cast<double>(hi))));
}

__global__ void init_sigmoid_table_kernel(double *table, float2 *table2, float4 *gelu_table, double2 *gelu_dtable,
                                          float2 *gelu_tail)
{
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536u) return;
    if (i < static_cast<uint32_t>(mx::kGeluTabN)) {
        // the GEGLU fast path's entry i: t = |g| of pattern kGeluTabLo + i - 1
        // (entry 0: every t below the first, taken as 0)
        const double t = i == 0 ? 0.0 : static_cast<double>(__uint_as_float((mx::kGeluTabLo + i - 1u) << 16));
        const double q = t * exp(-0.5 * t * t) * 0.39894228040143267794;   // t phi(t)
        gelu_tail[i] = make_float2(__double2float_rn(i == 0 ? 0.5 : mx::normal_cdf_double(-t)),
                                   __double2float_rn(q));
    }
    const float gf = __uint_as_float(i << 16);
    const double g = static_cast<double>(gf);
    const double s = mx::sigmoid_double(gf);  // 1 / (1 + e^-g)
    table[i] = s;
    table2[i] = float_pair(s);
    const double phi = mx::normal_cdf_double(g), dgelu = mx::gelu_grad_double(g);
    const float2 p = float_pair(phi), d = float_pair(dgelu);
    gelu_table[i] = make_float4(p.x, p.y, d.x, d.y);
    gelu_dtable[i] = make_double2(phi, dgelu);
}

__global__ void selftest_wait_kernel(unsigned *status, long long limit)
{
    __shared__ uint64_t bar;
    const uint32_t b = mx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        mx::mbar_init(b, 1);
        mx::fence_barrier_init();
    }
    __syncthreads();
    // nobody ever arrives: phase 0 never completes
    if (!mx::mbar_wait_bounded(b, 0u, limit)) atomicOr(status, mx::kStatusSelftestWait);
}

// The fast-path activation factors for every bf16 gate value, computed by the
// same device functions the tile kernels inline (on pairs of adjacent
// patterns): out[k * 65536 + g] for k = 0 sigmoid, 1 silu, 2 1-sigmoid,
// 3 w = 1 + g(1-sigmoid), 4 silu' = sigmoid * w, 5 2^120 e^g (the factor of
// the wide-range values for gates below the fast range).
__global__ void selftest_activation_kernel(float *out)
{
    const uint32_t i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= 65536u) return;
    const uint64_t G = mx::f2(__uint_as_float(i << 16), __uint_as_float((i + 1) << 16));
    uint64_t T;
    const uint64_t S = mx::sigmoid2(G, T, 1.0f);
    const uint64_t SN = mx::mul2(T, S);
    const uint64_t W = mx::fma2(G, SN, mx::f2(1.0f, 1.0f));
    const uint64_t V[6] = {S, mx::silu2_up(G), SN, W, mx::mul2(S, W), mx::exp_far2(G)};
    for (int k = 0; k < 6; ++k) {
        out[k * 65536 + i] = mx::f2lo(V[k]);
        out[k * 65536 + i + 1] = mx::f2hi(V[k]);
    }
}

// The GEGLU fast paths' gate-only factors for every bf16 pattern g (pairs of
// consecutive patterns per thread), computed by the device functions the
// tile kernels inline: out[k * 65536 + g] for k = 0 Phi(g), 1 gelu(g) =
// g Phi(g) as the forward forms it (the product (g * 1) Phi), 2 gelu'(g) =
// Phi(g) + g phi(g), from the tail table; 3 Phi(g) and 4 gelu'(g) from the
// rational tail.
__global__ void selftest_activation_gelu_kernel(float *out, const float2 *gelu_tail)
{
    mx::gelu_tail_fill<true>(gelu_tail);
    mx::gelu_tail_fill<false>(gelu_tail);
    __syncthreads();
    const uint32_t i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= 65536u) return;
    const uint32_t gw = i | ((i + 1) << 16);
    uint64_t E, DG, DU, DGP, DUP;
    mx::geglu_grads2(0x3F803F80u, gw, 0x3F803F80u, DG, DU);     // dh = u = 1: DG = gelu'(g)
    mx::geglu_grads2_poly(0x3F803F80u, gw, 0x3F803F80u, DGP, DUP);
    const uint64_t V[5] = {mx::normal_cdf2(gw), mx::geglu_h2(gw, 0x3F803F80u), DG, mx::normal_cdf2_poly(gw, E), DGP};
    for (int k = 0; k < 5; ++k) {
        out[k * 65536 + i] = mx::f2lo(V[k]);
        out[k * 65536 + i + 1] = mx::f2hi(V[k]);
    }
}

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::atomic<bool> ready{false};
    double *table = nullptr;
    float2 *table2 = nullptr;
    float4 *gelu_table = nullptr;
    double2 *gelu_dtable = nullptr;
    float2 *gelu_tail = nullptr;
    unsigned *status = nullptr;
    unsigned long long *fallbacks = nullptr;
    int sms = 0;
    long long wait_limit = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_init_mutex;

mxfp8_status ensure_device(cudaStream_t stream, int *dev_out, DeviceState **state)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP8_ERR_DEVICE;
    DeviceState &d = g_dev[dev];
    *dev_out = dev;
    *state = &d;
    if (d.ready.load(std::memory_order_acquire)) return MXFP8_OK;
    std::lock_guard<std::mutex> lock(g_init_mutex);
    if (d.ready.load(std::memory_order_acquire)) return MXFP8_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
        return MXFP8_ERR_CAPTURE;
    int major = 0, minor = 0, sms = 0, clock_khz = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MXFP8_ERR_DEVICE;
    if (major != 10 || minor != 3) return MXFP8_ERR_DEVICE;  // built for sm_103a only
    if (cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess || clock_khz <= 0)
        clock_khz = 2000000;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sig_table) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.table = static_cast<double *>(p);
    if (cudaGetSymbolAddress(&p, g_sig2_table) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.table2 = static_cast<float2 *>(p);
    if (cudaGetSymbolAddress(&p, g_gelu_table) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.gelu_table = static_cast<float4 *>(p);
    if (cudaGetSymbolAddress(&p, g_gelu_dtable) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.gelu_dtable = static_cast<double2 *>(p);
    if (cudaGetSymbolAddress(&p, g_gelu_tail) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.gelu_tail = static_cast<float2 *>(p);
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.status = static_cast<unsigned *>(p);
    if (cudaGetSymbolAddress(&p, g_fallbacks) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.fallbacks = static_cast<unsigned long long *>(p);
    init_sigmoid_table_kernel<<<256, 256, 0, stream>>>(d.table, d.table2, d.gelu_table, d.gelu_dtable, d.gelu_tail);
    if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_DEVICE;
    if (cudaMemsetAsync(d.status, 0, sizeof(unsigned), stream) != cudaSuccess ||
        cudaMemsetAsync(d.fallbacks, 0, sizeof(unsigned long long), stream) != cudaSuccess)
        return MXFP8_ERR_DEVICE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MXFP8_ERR_DEVICE;
    d.sms = sms;
    d.wait_limit = static_cast<long long>(clock_khz) * 1000;  // about one second of SM clock
    d.ready.store(true, std::memory_order_release);
    return MXFP8_OK;
}

// --------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// bf16 (rows, cols) with row pitch ld elements, boxes of box_rows x 64 cols,
// 128-byte swizzle, zero fill outside the tensor.
bool make_bf16_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld,
                   int box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(mx::kBoxN), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// --------------------------------------------------------------- checking
struct Region {        // rows of `width` bytes, `pitch` bytes apart
    uintptr_t base;
    int64_t rows, width, pitch;
    bool used;
};

Region region(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t elem)
{
    return Region{reinterpret_cast<uintptr_t>(p), rows, cols * elem, ld * elem, p != nullptr};
}

int64_t floordiv(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Do two strided byte regions share a byte?  Exact when the pitches are
// equal, conservative (extent overlap) otherwise.
bool regions_overlap(const Region &a, const Region &b)
{
    if (!a.used || !b.used || a.rows <= 0 || b.rows <= 0) return false;
    const int64_t a_end = static_cast<int64_t>(a.base) + (a.rows - 1) * a.pitch + a.width;
    const int64_t b_end = static_cast<int64_t>(b.base) + (b.rows - 1) * b.pitch + b.width;
    if (a_end <= static_cast<int64_t>(b.base) || b_end <= static_cast<int64_t>(a.base)) return false;
    if (a.pitch != b.pitch || a.width > a.pitch || b.width > b.pitch) return true;
    const int64_t L = a.pitch;
    const int64_t d = static_cast<int64_t>(b.base) - static_cast<int64_t>(a.base);
    const int64_t k = floordiv(d, L);
    const int64_t r = d - k * L;  // 0 <= r < L
    // B row j starts r bytes into A's pitch window j + k
    const bool same_window = r < a.width && k < a.rows && k + b.rows > 0;
    const bool next_window = r + b.width > L && k + 1 < a.rows && k + 1 + b.rows > 0;
    return same_window || next_window;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }

// extent check: (rows - 1) * ld + cols fits in int64 (and as bytes * elem)
bool extent_ok(int64_t rows, int64_t cols, int64_t ld, int64_t elem)
{
    int64_t t;
    if (!mul_ok(rows, ld, &t)) return false;
    if (__builtin_add_overflow(t, cols, &t)) return false;
    return mul_ok(t, elem, &t);
}

constexpr int64_t kMaxDim = 0x7FFFFF00LL;  // TMA coordinates are signed 32-bit

struct Spec {
    int op;               // mx::kQuant / kFwd / kBwd
    int mode;             // MXFP8_ROWWISE / COLWISE / BOTH, possibly | MXFP8_BLOCKED_SCALES
    int64_t M, N;
    const void *in[3];
    int64_t ld_in[3];
    uint8_t *q_row[2], *s_row[2], *q_col[2], *s_col[2];
    int64_t ld_qrow, ld_srow, ld_qcol, ld_scol;
    int64_t group_rows, group_stride;
    uint16_t *h;          // forward with the bf16 activation as an output
    int64_t ld_h;
    bool with_h;
    int act;              // mx::kSilu / kGelu (the fused ops)
    const int32_t *group_end;   // per-group blocked scales: token groups' end rows (device)
    int64_t num_groups;
    bool per_expert;      // 3D with blocked scales: one blocked matrix per expert
};

// Bytes of a scale matrix of R rows and C columns in the blocked layout
// (padded to multiples of 128 rows and 4 columns).
int64_t blocked_bytes(int64_t R, int64_t C) { return (R + 127) / 128 * 128 * ((C + 3) / 4 * 4); }

// Bytes of the row- and column-scale buffers in the blocked layouts: plain,
// per token group (M-groups / K-groups: (ceil(M/128) + G) 128-row tiles of
// the row scales, (ceil(M/128) + G) 4-column tiles of the column scales) or
// per expert (3D, group_rows rows an expert).
int64_t row_scale_bytes(const Spec &s)
{
    if (s.group_end) return ((s.M + 127) / 128 + s.num_groups) * 128 * ((s.N / 32 + 3) / 4 * 4);
    if (s.per_expert) return s.M / s.group_rows * blocked_bytes(s.group_rows, s.N / 32);
    return blocked_bytes(s.M, s.N / 32);
}

int64_t col_scale_bytes(const Spec &s)
{
    if (s.group_end) return (s.N + 127) / 128 * 128 * (((s.M + 127) / 128 + s.num_groups) * 4);
    if (s.per_expert) return s.M / s.group_rows * blocked_bytes(s.N, s.group_rows / 32);
    return blocked_bytes(s.N, s.M / 32);
}

mxfp8_status validate(const Spec &s)
{
    const int nin = s.op == mx::kQuant ? 1 : (s.op == mx::kFwd ? 2 : 3);
    const int nout = s.op == mx::kBwd ? 2 : 1;
    if ((s.mode & ~(3 | MXFP8_BLOCKED_SCALES)) != 0 || (s.mode & 3) == 0) return MXFP8_ERR_MODE;
    const bool blocked = (s.mode & MXFP8_BLOCKED_SCALES) != 0;
    if (blocked && s.group_stride != 0 && !s.per_expert) return MXFP8_ERR_MODE;
    if (s.act != mx::kSilu && s.act != mx::kGelu) return MXFP8_ERR_MODE;
    if (s.M < 0 || s.N < 0) return MXFP8_ERR_SHAPE;
    if (s.group_end || s.num_groups != 0) {          // per token group
        if (s.num_groups < 1 || s.num_groups > mx::kMaxGroups) return MXFP8_ERR_SHAPE;
        if (!s.group_end) return MXFP8_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(s.group_end) & 3u) != 0) return MXFP8_ERR_ALIGN;
        if (s.M > 0x7FFFFFFFLL - 128 * (mx::kMaxGroups + 1)) return MXFP8_ERR_SHAPE;   // 32-bit shifts
    }
    if (s.M == 0 || s.N == 0) return MXFP8_OK;
    if (s.M > kMaxDim || s.N > kMaxDim) return MXFP8_ERR_SHAPE;
    // the kernels walk their tiles (at least 96 x 128 elements each) with
    // 32-bit counters
    if ((s.M + 95) / 96 * ((s.N + 127) / 128) > 0x7FFFFFFFLL - 4096) return MXFP8_ERR_SHAPE;
    const bool row = s.mode & 1, col = s.mode & 2;
    if (s.per_expert && blocked && s.group_rows % 32 != 0) return MXFP8_ERR_SHAPE;
    if (row && s.N % 32 != 0) return MXFP8_ERR_SHAPE;
    if (col && s.M % 32 != 0) return MXFP8_ERR_SHAPE;
    for (int i = 0; i < nin; ++i) {
        if (!s.in[i]) return MXFP8_ERR_NULL;
    }
    if (s.with_h) {
        if (!row) return MXFP8_ERR_MODE;
        if (!s.h) return MXFP8_ERR_NULL;
        if (s.ld_h < s.N) return MXFP8_ERR_LD;
        if (!extent_ok(s.M, s.N, s.ld_h, 2)) return MXFP8_ERR_SHAPE;
        if (!aligned16(s.h) || (s.ld_h * 2) % 16 != 0) return MXFP8_ERR_ALIGN;
    }
    for (int o = 0; o < nout; ++o) {
        if (row && (!s.q_row[o] || !s.s_row[o])) return MXFP8_ERR_NULL;
        if (col && (!s.q_col[o] || !s.s_col[o])) return MXFP8_ERR_NULL;
    }
    for (int i = 0; i < nin; ++i) {
        if (s.ld_in[i] < s.N) return MXFP8_ERR_LD;
        if (!extent_ok(s.M, s.N, s.ld_in[i], 2) || s.ld_in[i] > (int64_t(1) << 38)) return MXFP8_ERR_SHAPE;
        if (!aligned16(s.in[i]) || (s.ld_in[i] * 2) % 16 != 0) return MXFP8_ERR_ALIGN;
    }
    if (row) {
        if (s.ld_qrow < s.N || (!blocked && s.ld_srow < s.N / 32)) return MXFP8_ERR_LD;
        if (!extent_ok(s.M, s.N, s.ld_qrow, 1) || (!blocked && !extent_ok(s.M, s.N / 32, s.ld_srow, 1)))
            return MXFP8_ERR_SHAPE;
        if (s.ld_qrow % 16 != 0) return MXFP8_ERR_ALIGN;
        for (int o = 0; o < nout; ++o) {
            if (!aligned16(s.q_row[o])) return MXFP8_ERR_ALIGN;
            if (blocked && (reinterpret_cast<uintptr_t>(s.s_row[o]) & 3u) != 0) return MXFP8_ERR_ALIGN;
        }
    }
    if (col) {
        if (s.group_stride == 0) {  // 2D column-major
            if (s.ld_qcol < s.M || (!blocked && s.ld_scol < s.N)) return MXFP8_ERR_LD;
            if (!extent_ok(s.N, s.M, s.ld_qcol, 1) || (!blocked && !extent_ok(s.M / 32, s.N, s.ld_scol, 1)))
                return MXFP8_ERR_SHAPE;
        }
        if (s.ld_qcol % 16 != 0) return MXFP8_ERR_ALIGN;
        for (int o = 0; o < nout; ++o)
            if (!aligned16(s.q_col[o])) return MXFP8_ERR_ALIGN;
    }
    // overlap: outputs against inputs and against each other
    Region ins[3], outs[8];
    int n_outs = 0;
    for (int i = 0; i < nin; ++i) ins[i] = region(s.in[i], s.M, s.N, s.ld_in[i], 2);
    if (s.with_h) outs[n_outs++] = region(s.h, s.M, s.N, s.ld_h, 2);
    for (int o = 0; o < nout; ++o) {
        if (row) {
            outs[n_outs++] = region(s.q_row[o], s.M, s.N, s.ld_qrow, 1);
            if (blocked) {
                const int64_t b = row_scale_bytes(s);
                outs[n_outs++] = region(s.s_row[o], 1, b, b, 1);
            } else {
                outs[n_outs++] = region(s.s_row[o], s.M, s.N / 32, s.ld_srow, 1);
            }
        }
        if (col) {
            if (s.group_stride == 0) {
                outs[n_outs++] = region(s.q_col[o], s.N, s.M, s.ld_qcol, 1);
            } else {  // 3D: E * K rows of N bytes
                const int64_t E = s.M / s.group_rows;
                outs[n_outs++] = region(s.q_col[o], E * s.N, s.group_rows, s.ld_qcol, 1);
            }
            if (blocked) {
                const int64_t b = col_scale_bytes(s);
                outs[n_outs++] = region(s.s_col[o], 1, b, b, 1);
            } else {
                outs[n_outs++] = region(s.s_col[o], s.M / 32, s.N, s.ld_scol, 1);
            }
        }
    }
    const Region groups = region(s.group_end, 1, 4 * s.num_groups, 4 * s.num_groups, 1);
    for (int a = 0; a < n_outs; ++a) {
        for (int i = 0; i < nin; ++i)
            if (regions_overlap(outs[a], ins[i])) return MXFP8_ERR_OVERLAP;
        if (s.group_end && regions_overlap(outs[a], groups)) return MXFP8_ERR_OVERLAP;
        for (int b = a + 1; b < n_outs; ++b)
            if (regions_overlap(outs[a], outs[b])) return MXFP8_ERR_OVERLAP;
    }
    return MXFP8_OK;
}

mxfp8_status run(const Spec &s, void *stream_ptr)
{
    mxfp8_status st = validate(s);
    if (st != MXFP8_OK || s.M == 0 || s.N == 0) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int dev = -1;
    DeviceState *d = nullptr;
    st = ensure_device(stream, &dev, &d);
    if (st != MXFP8_OK) return st;
    if (!get_encoder()) return MXFP8_ERR_DEVICE;
    const int nin = s.op == mx::kQuant ? 1 : (s.op == mx::kFwd ? 2 : 3);
    const int mode = s.mode & 3;
    // per-group blocked scales run their own instantiations
    const bool grouped = (s.mode & MXFP8_BLOCKED_SCALES) != 0 &&
                         (s.group_end != nullptr || (s.per_expert && s.group_rows / 32 > 0));
    const mx::LaunchShape shape = mx::launch_shape(s.op, mode, s.op == mx::kQuant ? mx::kSilu : s.act, grouped);
    const int tm = shape.tile_rows;
    CUtensorMap maps[3];
    std::memset(maps, 0, sizeof(maps));
    for (int i = 0; i < 3; ++i) {
        const int src = i < nin ? i : 0;
        if (!make_bf16_map(&maps[i], s.in[src], s.M, s.N, s.ld_in[src], tm)) return MXFP8_ERR_ALIGN;
    }
    KernelArgs a;
    std::memset(&a, 0, sizeof(a));
    a.M = s.M;
    a.N = s.N;
    a.tiles_n = (s.N + mx::kTileN - 1) / mx::kTileN;
    a.num_tiles = ((s.M + tm - 1) / tm) * a.tiles_n;
    for (int o = 0; o < 2; ++o) {
        a.q_row[o] = s.q_row[o];
        a.s_row[o] = s.s_row[o];
        a.q_col[o] = s.q_col[o];
        a.s_col[o] = s.s_col[o];
    }
    a.ld_qrow = s.ld_qrow;
    a.ld_srow = s.ld_srow;
    a.ld_qcol = s.ld_qcol;
    a.ld_scol = s.ld_scol;
    a.group_rows = s.group_rows > 0 ? s.group_rows : s.M;
    a.group_stride = s.group_stride;
    // blocked scales: 128 x 4 tiles of the (M, N/32) row scales and of the
    // (N, M/32) column scales
    a.blocked = (s.mode & MXFP8_BLOCKED_SCALES) != 0;
    a.h_out = s.with_h ? s.h : nullptr;
    a.ld_h = s.ld_h;
    a.wide_h = s.with_h && (reinterpret_cast<uintptr_t>(s.h) & 31u) == 0 && (s.ld_h * 2) % 32 == 0;
    a.srow_tiles_c = (s.N / 32 + 3) / 4;
    a.scol_tiles_c = (s.M / 32 + 3) / 4;
    if (a.blocked && s.group_end) {           // M-groups row scales, K-groups column scales
        a.group_end = s.group_end;
        a.num_groups = static_cast<int>(s.num_groups);
        a.scol_tiles_c = (s.M + 127) / 128 + s.num_groups;
    } else if (a.blocked && s.per_expert) {   // one blocked matrix per expert
        a.uni_blocks = s.group_rows / 32;
        a.uni_r = (s.group_rows + 127) / 128 * 128 - s.group_rows;
        a.uni_crow = (s.N + 127) / 128 * 128;
        a.uni_c = -(s.group_rows / 32);
        a.scol_tiles_c = (s.group_rows / 32 + 3) / 4;
    }
    // whole 32-byte output blocks can go out as single 256-bit stores when
    // every block start is 32-byte aligned
    a.wide_row = (s.ld_qrow % 32) == 0;
    a.wide_col = (s.ld_qcol % 32) == 0 && (s.group_stride % 32) == 0;
    // a group of column tiles leaves its row scales as one 4*group-byte store
    // per row when rows are aligned to that
    const int64_t sgrp = 4 * static_cast<int64_t>(shape.group);
    a.wide_srow = (s.ld_srow % sgrp) == 0;
    for (int o = 0; o < 2; ++o) {
        if (s.s_row[o] && (reinterpret_cast<uintptr_t>(s.s_row[o]) % static_cast<uintptr_t>(sgrp)) != 0)
            a.wide_srow = 0;
        if (s.q_row[o] && (reinterpret_cast<uintptr_t>(s.q_row[o]) & 31u) != 0) a.wide_row = 0;
        if (s.q_col[o] && (reinterpret_cast<uintptr_t>(s.q_col[o]) & 31u) != 0) a.wide_col = 0;
    }
    a.sig_table = d->table;
    a.sig2_table = d->table2;
    a.gelu_table = d->gelu_table;
    a.gelu_dtable = d->gelu_dtable;
    a.gelu_tail = d->gelu_tail;
    a.status = d->status;
    a.fallbacks = d->fallbacks;
    a.wait_limit = d->wait_limit;
    // CTAs walk groups of `group` consecutive column tiles
    const int64_t supers = ((s.M + tm - 1) / tm) * ((a.tiles_n + shape.group - 1) / shape.group);
    const int64_t slots = static_cast<int64_t>(d->sms) * shape.ctas_per_sm;
    const int grid = static_cast<int>(supers < slots ? supers : slots);
    cudaError_t e;
    switch (s.op) {
    case mx::kQuant:
        e = grouped ? mx::launch_quant_grouped(mode, maps, a, grid, stream, dev)
                    : mx::launch_quant(mode, maps, a, grid, stream, dev);
        break;
    case mx::kFwd:
        if (s.act == mx::kGelu)
            e = grouped ? mx::launch_fwd_gelu_grouped(mode, maps, a, grid, stream, dev)
                        : mx::launch_fwd_gelu(mode, maps, a, grid, stream, dev);
        else
            e = grouped ? mx::launch_fwd_grouped(mode, maps, a, grid, stream, dev)
                        : mx::launch_fwd(mode, maps, a, grid, stream, dev);
        break;
    default:
        if (s.act == mx::kGelu)
            e = grouped ? mx::launch_bwd_gelu_grouped(mode, maps, a, grid, stream, dev)
                        : mx::launch_bwd_gelu(mode, maps, a, grid, stream, dev);
        else
            e = grouped ? mx::launch_bwd_grouped(mode, maps, a, grid, stream, dev)
                        : mx::launch_bwd(mode, maps, a, grid, stream, dev);
        break;
    }
    return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

Spec blank(int op, int mode, int64_t M, int64_t N)
{
    Spec s;
    std::memset(&s, 0, sizeof(s));
    s.op = op;
    s.mode = mode;
    s.M = M;
    s.N = N;
    return s;
}

// The fused forward's and backward's arguments (activation `act`), as the
// entry points take them.
Spec fwd_spec(int act, const uint16_t *gate, const uint16_t *up, int64_t ld_in, int64_t M, int64_t N, int mode,
              uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow, uint8_t *q_col, int64_t ld_qcol,
              uint8_t *s_col, int64_t ld_scol)
{
    Spec s = blank(mx::kFwd, mode, M, N);
    s.act = act;
    s.in[0] = gate;
    s.in[1] = up;
    s.ld_in[0] = s.ld_in[1] = ld_in;
    s.q_row[0] = q_row;
    s.s_row[0] = s_row;
    s.q_col[0] = q_col;
    s.s_col[0] = s_col;
    s.ld_qrow = ld_qrow;
    s.ld_srow = ld_srow;
    s.ld_qcol = ld_qcol;
    s.ld_scol = ld_scol;
    return s;
}

Spec bwd_spec(int act, const uint16_t *dh, int64_t ld_dh, const uint16_t *gate, const uint16_t *up, int64_t ld_in,
              int64_t M, int64_t N, int mode, uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow, uint8_t *dg_srow,
              uint8_t *du_srow, int64_t ld_srow, uint8_t *dg_col, uint8_t *du_col, int64_t ld_qcol,
              uint8_t *dg_scol, uint8_t *du_scol, int64_t ld_scol)
{
    Spec s = blank(mx::kBwd, mode, M, N);
    s.act = act;
    s.in[0] = dh;
    s.in[1] = gate;
    s.in[2] = up;
    s.ld_in[0] = ld_dh;
    s.ld_in[1] = s.ld_in[2] = ld_in;
    s.q_row[0] = dg_row;
    s.q_row[1] = du_row;
    s.s_row[0] = dg_srow;
    s.s_row[1] = du_srow;
    s.q_col[0] = dg_col;
    s.q_col[1] = du_col;
    s.s_col[0] = dg_scol;
    s.s_col[1] = du_scol;
    s.ld_qrow = ld_qrow;
    s.ld_srow = ld_srow;
    s.ld_qcol = ld_qcol;
    s.ld_scol = ld_scol;
    return s;
}

}  // namespace

extern "C" {

const char *mxfp8_status_str(mxfp8_status s)
{
    switch (s) {
    case MXFP8_OK: return "MXFP8_OK";
    case MXFP8_ERR_NULL: return "MXFP8_ERR_NULL: a required pointer is NULL";
    case MXFP8_ERR_SHAPE: return "MXFP8_ERR_SHAPE: invalid or unsupported shape";
    case MXFP8_ERR_ALIGN: return "MXFP8_ERR_ALIGN: misaligned pointer or leading dimension";
    case MXFP8_ERR_LD: return "MXFP8_ERR_LD: leading dimension too small";
    case MXFP8_ERR_MODE: return "MXFP8_ERR_MODE: scale mode must be 1, 2 or 3 (optionally | MXFP8_BLOCKED_SCALES)";
    case MXFP8_ERR_OVERLAP: return "MXFP8_ERR_OVERLAP: an output overlaps an input or another output";
    case MXFP8_ERR_LAUNCH: return "MXFP8_ERR_LAUNCH: kernel launch failed";
    case MXFP8_ERR_DEVICE: return "MXFP8_ERR_DEVICE: no usable sm_103 device or device set-up failed";
    case MXFP8_ERR_CAPTURE: return "MXFP8_ERR_CAPTURE: first use of a device inside a stream capture";
    }
    return "MXFP8_ERR_UNKNOWN";
}

int mxfp8_version(void) { return 100; }

mxfp8_status mxfp8_init(void *stream)
{
    int dev;
    DeviceState *d;
    return ensure_device(static_cast<cudaStream_t>(stream), &dev, &d);
}

mxfp8_status mxfp8_quant_2d(const uint16_t *x, int64_t ld_x, int64_t M, int64_t N, int mode,
                            uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                            uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                            void *stream)
{
    Spec s = blank(mx::kQuant, mode, M, N);
    s.in[0] = x;
    s.ld_in[0] = ld_x;
    s.q_row[0] = q_row;
    s.s_row[0] = s_row;
    s.q_col[0] = q_col;
    s.s_col[0] = s_col;
    s.ld_qrow = ld_qrow;
    s.ld_srow = ld_srow;
    s.ld_qcol = ld_qcol;
    s.ld_scol = ld_scol;
    return run(s, stream);
}

mxfp8_status mxfp8_swiglu_fwd(const uint16_t *gate, const uint16_t *up, int64_t ld_in, int64_t M,
                              int64_t N, int mode, uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                              int64_t ld_srow, uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col,
                              int64_t ld_scol, void *stream)
{
    return run(fwd_spec(mx::kSilu, gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow, q_col, ld_qcol,
                        s_col, ld_scol),
               stream);
}

mxfp8_status mxfp8_swiglu_fwd_with_h(const uint16_t *gate, const uint16_t *up, int64_t ld_in, int64_t M,
                                     int64_t N, int mode, uint16_t *h, int64_t ld_h, uint8_t *q_row,
                                     int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow, uint8_t *q_col,
                                     int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol, void *stream)
{
    Spec s = fwd_spec(mx::kSilu, gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow, q_col, ld_qcol, s_col,
                      ld_scol);
    s.with_h = true;
    s.h = h;
    s.ld_h = ld_h;
    return run(s, stream);
}

mxfp8_status mxfp8_swiglu_bwd(const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                              const uint16_t *up, int64_t ld_in, int64_t M, int64_t N, int mode,
                              uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow, uint8_t *dg_srow,
                              uint8_t *du_srow, int64_t ld_srow, uint8_t *dg_col, uint8_t *du_col,
                              int64_t ld_qcol, uint8_t *dg_scol, uint8_t *du_scol, int64_t ld_scol,
                              void *stream)
{
    return run(bwd_spec(mx::kSilu, dh, ld_dh, gate, up, ld_in, M, N, mode, dg_row, du_row, ld_qrow, dg_srow, du_srow,
                        ld_srow, dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol),
               stream);
}

mxfp8_status mxfp8_geglu_fwd(const uint16_t *gate, const uint16_t *up, int64_t ld_in, int64_t M,
                              int64_t N, int mode, uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                              int64_t ld_srow, uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col,
                              int64_t ld_scol, void *stream)
{
    return run(fwd_spec(mx::kGelu, gate, up, ld_in, M, N, mode, q_row, ld_qrow, s_row, ld_srow, q_col, ld_qcol,
                        s_col, ld_scol),
               stream);
}

mxfp8_status mxfp8_geglu_bwd(const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                              const uint16_t *up, int64_t ld_in, int64_t M, int64_t N, int mode,
                              uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow, uint8_t *dg_srow,
                              uint8_t *du_srow, int64_t ld_srow, uint8_t *dg_col, uint8_t *du_col,
                              int64_t ld_qcol, uint8_t *dg_scol, uint8_t *du_scol, int64_t ld_scol,
                              void *stream)
{
    return run(bwd_spec(mx::kGelu, dh, ld_dh, gate, up, ld_in, M, N, mode, dg_row, du_row, ld_qrow, dg_srow, du_srow,
                        ld_srow, dg_col, du_col, ld_qcol, dg_scol, du_scol, ld_scol),
               stream);
}

mxfp8_status mxfp8_quant_3d_colwise(const uint16_t *x, int64_t E, int64_t N, int64_t K, uint8_t *q,
                                    uint8_t *s, void *stream)
{
    if (E < 0 || N < 0 || K < 0) return MXFP8_ERR_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MXFP8_OK;
    if (N % 32 != 0) return MXFP8_ERR_SHAPE;
    int64_t rows;
    if (!mul_ok(E, N, &rows) || rows > kMaxDim || K > kMaxDim) return MXFP8_ERR_SHAPE;
    if (K % 8 != 0) return MXFP8_ERR_ALIGN;
    int64_t slab;
    if (!mul_ok(N, K, &slab)) return MXFP8_ERR_SHAPE;
    Spec sp = blank(mx::kQuant, MXFP8_COLWISE, rows, K);
    sp.in[0] = x;
    sp.ld_in[0] = K;
    sp.q_col[0] = q;
    sp.s_col[0] = s;
    sp.ld_qcol = N;       // within an expert: element (n, k) at k * N + n
    sp.ld_scol = K;       // scales (E * N/32, K) row-major
    sp.group_rows = N;
    sp.group_stride = slab;
    return run(sp, stream);
}

mxfp8_status mxfp8_quant_3d(const uint16_t *x, int64_t E, int64_t N, int64_t K, int mode, uint8_t *q_row,
                            uint8_t *s_row, uint8_t *q_col, uint8_t *s_col, void *stream)
{
    if ((mode & ~(3 | MXFP8_BLOCKED_SCALES)) != 0 || (mode & 3) == 0) return MXFP8_ERR_MODE;
    if (E < 0 || N < 0 || K < 0) return MXFP8_ERR_SHAPE;
    if (E == 0 || N == 0 || K == 0) return MXFP8_OK;
    if ((mode & MXFP8_COLWISE) && N % 32 != 0) return MXFP8_ERR_SHAPE;
    int64_t rows;
    if (!mul_ok(E, N, &rows) || rows > kMaxDim || K > kMaxDim) return MXFP8_ERR_SHAPE;
    if (K % 8 != 0) return MXFP8_ERR_ALIGN;
    int64_t slab;
    if (!mul_ok(N, K, &slab)) return MXFP8_ERR_SHAPE;
    Spec sp = blank(mx::kQuant, mode, rows, K);
    sp.in[0] = x;
    sp.ld_in[0] = K;
    sp.q_row[0] = q_row;  // (E, N, K) row-major: the (E * N, K) matrix
    sp.s_row[0] = s_row;
    sp.ld_qrow = K;
    sp.ld_srow = K / 32;
    sp.q_col[0] = q_col;
    sp.s_col[0] = s_col;
    sp.ld_qcol = N;
    sp.ld_scol = K;
    sp.group_rows = N;
    sp.group_stride = (mode & MXFP8_COLWISE) ? slab : 0;
    sp.per_expert = (mode & MXFP8_BLOCKED_SCALES) != 0;
    if (sp.group_stride == 0 && sp.per_expert && N % 32 != 0) return MXFP8_ERR_SHAPE;
    return run(sp, stream);
}

mxfp8_status mxfp8_quant_2d_grouped(const uint16_t *x, int64_t ld_x, int64_t M, int64_t N, int mode,
                                    const int32_t *group_end, int64_t num_groups, uint8_t *q_row,
                                    int64_t ld_qrow, uint8_t *s_row, uint8_t *q_col, int64_t ld_qcol,
                                    uint8_t *s_col, void *stream)
{
    Spec s = blank(mx::kQuant, mode | MXFP8_BLOCKED_SCALES, M, N);
    if ((mode & ~(3 | MXFP8_BLOCKED_SCALES)) != 0) return MXFP8_ERR_MODE;
    s.in[0] = x;
    s.ld_in[0] = ld_x;
    s.q_row[0] = q_row;
    s.s_row[0] = s_row;
    s.q_col[0] = q_col;
    s.s_col[0] = s_col;
    s.ld_qrow = ld_qrow;
    s.ld_qcol = ld_qcol;
    s.group_end = group_end;
    s.num_groups = num_groups;
    return run(s, stream);
}

mxfp8_status mxfp8_swiglu_fwd_grouped(const uint16_t *gate, const uint16_t *up, int64_t ld_in, int64_t M,
                                      int64_t N, int mode, int act, const int32_t *group_end,
                                      int64_t num_groups, uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                                      uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, void *stream)
{
    if ((mode & ~(3 | MXFP8_BLOCKED_SCALES)) != 0) return MXFP8_ERR_MODE;
    Spec s = fwd_spec(act, gate, up, ld_in, M, N, mode | MXFP8_BLOCKED_SCALES, q_row, ld_qrow, s_row, 0, q_col,
                      ld_qcol, s_col, 0);
    s.group_end = group_end;
    s.num_groups = num_groups;
    return run(s, stream);
}

mxfp8_status mxfp8_swiglu_bwd_grouped(const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                                      const uint16_t *up, int64_t ld_in, int64_t M, int64_t N, int mode,
                                      int act, const int32_t *group_end, int64_t num_groups,
                                      uint8_t *dg_row, uint8_t *du_row, int64_t ld_qrow, uint8_t *dg_srow,
                                      uint8_t *du_srow, uint8_t *dg_col, uint8_t *du_col, int64_t ld_qcol,
                                      uint8_t *dg_scol, uint8_t *du_scol, void *stream)
{
    if ((mode & ~(3 | MXFP8_BLOCKED_SCALES)) != 0) return MXFP8_ERR_MODE;
    Spec s = bwd_spec(act, dh, ld_dh, gate, up, ld_in, M, N, mode | MXFP8_BLOCKED_SCALES, dg_row, du_row, ld_qrow,
                      dg_srow, du_srow, 0, dg_col, du_col, ld_qcol, dg_scol, du_scol, 0);
    s.group_end = group_end;
    s.num_groups = num_groups;
    return run(s, stream);
}

mxfp8_status mxfp8_device_status(uint32_t *flags, uint64_t *fallbacks, int reset, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev;
    DeviceState *d;
    mxfp8_status r = ensure_device(st, &dev, &d);
    if (r != MXFP8_OK) return r;
    unsigned f = 0;
    unsigned long long n = 0;
    if (cudaMemcpyAsync(&f, d->status, sizeof f, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(&n, d->fallbacks, sizeof n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MXFP8_ERR_DEVICE;
    if (reset) {
        if (cudaMemsetAsync(d->status, 0, sizeof(unsigned), st) != cudaSuccess ||
            cudaMemsetAsync(d->fallbacks, 0, sizeof(unsigned long long), st) != cudaSuccess)
            return MXFP8_ERR_DEVICE;
    }
    if (cudaStreamSynchronize(st) != cudaSuccess) return MXFP8_ERR_DEVICE;
    if (flags) *flags = f;
    if (fallbacks) *fallbacks = n;
    return MXFP8_OK;
}

mxfp8_status mxfp8_selftest_activation(float *out, void *stream)
{
    if (!out) return MXFP8_ERR_NULL;
    if (!aligned16(out)) return MXFP8_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev;
    DeviceState *d;
    mxfp8_status r = ensure_device(st, &dev, &d);
    if (r != MXFP8_OK) return r;
    selftest_activation_kernel<<<128, 256, 0, st>>>(out);
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

mxfp8_status mxfp8_selftest_activation_gelu(float *out, void *stream)
{
    if (!out) return MXFP8_ERR_NULL;
    if (!aligned16(out)) return MXFP8_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev;
    DeviceState *d;
    mxfp8_status r = ensure_device(st, &dev, &d);
    if (r != MXFP8_OK) return r;
    selftest_activation_gelu_kernel<<<128, 256, 0, st>>>(out, d->gelu_tail);
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

mxfp8_status mxfp8_selftest_wait_timeout(uint64_t limit_cycles, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev;
    DeviceState *d;
    mxfp8_status r = ensure_device(st, &dev, &d);
    if (r != MXFP8_OK) return r;
    const long long lim = limit_cycles > (1ull << 40) ? (1ll << 40) : static_cast<long long>(limit_cycles);
    selftest_wait_kernel<<<1, 32, 0, st>>>(d->status, lim);
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free forward: for callers that cannot call cudaMalloc at all
// (code running inside a host framework's fixed device-memory arena, or in
// a context where allocating is forbidden, such as between the start and end
// of a stream capture that must not record allocation nodes).  It takes the
// same arguments as mxfp8_swiglu_fwd but materialises the activation in a
// scratch buffer that the library itself reserves statically.
namespace {

// Scratch for the bf16 activation of one call: 8,388,608 elements (16 MiB),
// reserved in every device's global memory when the library is loaded and
// held until the process exits.  Every call of the entry point reuses it.
constexpr int64_t kNoAllocScratchElems = 8ll * 1024 * 1024;
static __device__ __align__(256) uint16_t g_noalloc_scratch[kNoAllocScratchElems];

// device address of the scratch, looked up once per device (host code must
// not pass the symbol itself: on the host it is only a stand-in)
uint16_t *g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

mxfp8_status noalloc_scratch_ptr(uint16_t **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MXFP8_ERR_DEVICE;
        g_noalloc_ptr[dev] = static_cast<uint16_t *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MXFP8_OK;
}

// h = bf16(silu(gate) * up) for one 8-column chunk per thread, written to the
// scratch with row pitch ld_h; every element takes the exact path, so the
// cast that follows sees the correctly rounded activation.
__global__ void swiglu_activation_kernel(const uint16_t *__restrict__ gate,
                                         const uint16_t *__restrict__ up, int64_t ld_in,
                                         int64_t M, int64_t N, uint16_t *__restrict__ h,
                                         int64_t ld_h, KernelArgs a)
{
    const int64_t chunks_n = (N + 7) / 8;
    const int64_t total = M * chunks_n;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / chunks_n;
        const int64_t c = (i - r * chunks_n) * 8;
        const uint16_t *g = gate + r * ld_in + c;
        const uint16_t *u = up + r * ld_in + c;
        uint16_t *o = h + r * ld_h + c;
        if (c + 8 <= N) {
            const uint4 gv = *reinterpret_cast<const uint4 *>(g);
            const uint4 uv = *reinterpret_cast<const uint4 *>(u);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
            uint32_t ow[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float h0 = mx::swiglu_h_exact(a.sig2_table, a.sig_table, mx::bf16lo(gw[p]), mx::bf16lo(uw[p]));
                const float h1 = mx::swiglu_h_exact(a.sig2_table, a.sig_table, mx::bf16hi(gw[p]), mx::bf16hi(uw[p]));
                ow[p] = mx::pack_bf16x2(h0, h1);
            }
            *reinterpret_cast<uint4 *>(o) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        } else {
            for (int64_t k = 0; c + k < N; ++k) {
                const float gf = __uint_as_float(static_cast<uint32_t>(g[k]) << 16);
                const float uf = __uint_as_float(static_cast<uint32_t>(u[k]) << 16);
                const float hv = mx::swiglu_h_exact(a.sig2_table, a.sig_table, gf, uf);
                o[k] = static_cast<uint16_t>(mx::pack_bf16x2(hv, 0.0f) & 0xFFFFu);
            }
        }
    }
}

}  // namespace

extern "C" mxfp8_status mxfp8_swiglu_fwd_noalloc(const uint16_t *gate, const uint16_t *up,
                                                 int64_t ld_in, int64_t M, int64_t N, int mode,
                                                 uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row,
                                                 int64_t ld_srow, uint8_t *q_col, int64_t ld_qcol,
                                                 uint8_t *s_col, int64_t ld_scol, void *stream)
{
    // the fused forward's argument rules apply unchanged
    Spec fs = blank(mx::kFwd, mode, M, N);
    fs.in[0] = gate;
    fs.in[1] = up;
    fs.ld_in[0] = fs.ld_in[1] = ld_in;
    fs.q_row[0] = q_row;
    fs.s_row[0] = s_row;
    fs.q_col[0] = q_col;
    fs.s_col[0] = s_col;
    fs.ld_qrow = ld_qrow;
    fs.ld_srow = ld_srow;
    fs.ld_qcol = ld_qcol;
    fs.ld_scol = ld_scol;
    mxfp8_status st = validate(fs);
    if (st != MXFP8_OK || M == 0 || N == 0) return st;
    const int64_t ld_h = (N + 7) / 8 * 8;  // 16-byte rows for the cast's TMA tiles
    if (M > kNoAllocScratchElems / ld_h) return MXFP8_ERR_SHAPE;  // beyond the static scratch
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = -1;
    DeviceState *d = nullptr;
    st = ensure_device(s, &dev, &d);
    if (st != MXFP8_OK) return st;
    uint16_t *h = nullptr;
    st = noalloc_scratch_ptr(&h);
    if (st != MXFP8_OK) return st;
    KernelArgs a;
    std::memset(&a, 0, sizeof(a));
    a.sig_table = d->table;
    a.sig2_table = d->table2;
    a.gelu_table = d->gelu_table;
    a.gelu_dtable = d->gelu_dtable;
    a.gelu_tail = d->gelu_tail;
    a.fallbacks = d->fallbacks;
    a.status = d->status;
    const int64_t chunks = M * ((N + 7) / 8);
    const int blocks = static_cast<int>(std::min<int64_t>((chunks + 255) / 256, int64_t(d->sms) * 8));
    swiglu_activation_kernel<<<blocks, 256, 0, s>>>(gate, up, ld_in, M, N, h, ld_h, a);
    if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_LAUNCH;
    // second pass: the standalone cast of the activation just written
    Spec qs = blank(mx::kQuant, mode, M, N);
    qs.in[0] = h;
    qs.ld_in[0] = ld_h;
    qs.q_row[0] = q_row;
    qs.s_row[0] = s_row;
    qs.q_col[0] = q_col;
    qs.s_col[0] = s_col;
    qs.ld_qrow = ld_qrow;
    qs.ld_srow = ld_srow;
    qs.ld_qcol = ld_qcol;
    qs.ld_scol = ld_scol;
    return run(qs, stream);
}
