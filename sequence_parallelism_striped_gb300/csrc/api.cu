// api.cu -- the C entry points of libstriped (declared in include/striped.h):
// argument validation, status codes, tensor-map construction, the host-side
// tile/critical-path model, the device status word and the wait control.
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace striped {

// The library's status word on every device that loads it (one per device,
// shared by every stream and caller on that device).
__device__ DeviceStatus g_status = {0};

// Per-device host state: the status word's address (looked up once) and the
// wait bound and test hook that striped_test_inject sets.
struct HostDeviceState {
    DeviceStatus *st = nullptr;
    unsigned long long limit_ns = kDefaultWaitLimitNs;
    int inject = kInjectNone;
};
static std::mutex g_state_mu;
static HostDeviceState g_state[kMaxDevices];

DeviceStatus *device_status() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_state_mu);
    if (!g_state[dev].st) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
        g_state[dev].st = static_cast<DeviceStatus *>(ptr);
    }
    return g_state[dev].st;
}

WaitCtl device_wait_ctl() {
    WaitCtl w{device_status(), kDefaultWaitLimitNs, kInjectNone};
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_state_mu);
        w.limit_ns = g_state[dev].limit_ns;
        w.inject = g_state[dev].inject;
    }
    return w;
}

static thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t err) {
    if (err == cudaSuccess) return STRIPED_OK;
    t_last_cuda_error = (int)err;
    return STRIPED_ERR_CUDA;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFnT)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [BH][N][L][D] tensor of `esize`-byte elements -> 4-D tiled tensor map,
// boxes of box_x elements x box_rows rows, 128-byte swizzle, zero fill.
static int make_map(CUtensorMap *map, CUtensorMapDataType dt, int64_t esize, const void *base, int64_t D,
                    int64_t L, int64_t N, int64_t BH, int64_t stripe_stride, int64_t stride_bh, int box_x,
                    int box_rows) {
    // the driver entry point is process-wide: resolved once, under a lock
    static std::mutex mu;
    static EncodeTiledFnT fn = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!fn) {
            void *ptr = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                             cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr)
                return cuda_status(e != cudaSuccess ? e : cudaErrorNotSupported);
            fn = reinterpret_cast<EncodeTiledFnT>(ptr);
        }
    }
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[3] = {(cuuint64_t)(D * esize), (cuuint64_t)(stripe_stride * esize),
                             (cuuint64_t)(stride_bh * esize)};
    cuuint32_t box[4] = {(cuuint32_t)box_x, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = (int)r;
        return STRIPED_ERR_CUDA;
    }
    return STRIPED_OK;
}

int make_bf16_map(CUtensorMap *map, const void *base, int64_t D, int64_t L, int64_t N, int64_t BH,
                  int64_t stripe_stride, int64_t stride_bh, int box_rows) {
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, D, L, N, BH, stripe_stride, stride_bh, 64,
                    box_rows);
}

int make_f32_map(CUtensorMap *map, const void *base, int64_t D, int64_t L, int64_t N, int64_t BH,
                 int64_t stripe_stride, int64_t stride_bh, int box_rows) {
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, D, L, N, BH, stripe_stride, stride_bh, 32,
                    box_rows);
}

// ---------------------------------------------------------------- validation
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_sizes(int64_t B, int64_t H, int64_t S, int64_t D, int N) {
    if (B < 1 || H < 1 || S < 1 || D < 1 || N < 1) return STRIPED_ERR_INVALID_ARG;
    if (S % N != 0) return STRIPED_ERR_INVALID_ARG;
    if (S > (1ll << 31) || B * H > (1ll << 31)) return STRIPED_ERR_UNSUPPORTED;
    return STRIPED_OK;
}

static bool valid_layout(int layout) {
    return layout == STRIPED_LAYOUT_STRIPED || layout == STRIPED_LAYOUT_CONTIGUOUS ||
           layout == STRIPED_LAYOUT_ZIGZAG;
}

static int check_attn(int64_t B, int64_t H, int64_t S, int64_t D, int N, int layout, int dtype) {
    int st = check_sizes(B, H, S, D, N);
    if (st) return st;
    if (!valid_layout(layout)) return STRIPED_ERR_INVALID_ARG;
    int64_t tile;
    if (dtype == STRIPED_BF16) {
        if (D != 128 && D != 64) return STRIPED_ERR_UNSUPPORTED;
        tile = kTcTile;
    } else if (dtype == STRIPED_FP32) {
        if (D % 8 != 0 || D > 128) return STRIPED_ERR_UNSUPPORTED;
        tile = kSimtTile;
    } else {
        return STRIPED_ERR_INVALID_ARG;
    }
    if (layout == STRIPED_LAYOUT_ZIGZAG) {
        // whole chunks of C = S/(2N) rows, each a whole number of tiles
        if (S % (2 * (int64_t)N) != 0) return STRIPED_ERR_INVALID_ARG;
        if ((S / (2 * (int64_t)N)) % tile != 0) return STRIPED_ERR_UNSUPPORTED;
    }
    return STRIPED_OK;
}

static AttnGeom full_geom(int64_t B, int64_t H, int64_t Hkv, int64_t S, int64_t D, int N, int layout,
                          float scale) {
    AttnGeom g{};  // seqs.n = 0: dense
    g.BH = B * H;
    g.G = H / Hkv;
    g.L = S / N;
    g.D = D;
    g.N = N;
    g.layout = layout;
    g.stride_bh = S * D;
    g.stripe_stride = g.L * D;
    g.lse_stride_bh = S;
    g.lse_stripe_stride = g.L;
    g.scale = scale;
    return g;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- device kernels (tiny)
// A device word that nothing ever sets: the self-test waits on it.
__device__ int g_selftest_flag = 0;

__global__ void selftest_wait_kernel(int64_t spins) {
    const volatile int *flag = &g_selftest_flag;
    for (int64_t it = 0; it < spins; ++it)
        if (*flag != 0) return;
    atomicExch(&g_status.error, STRIPED_ERR_TIMEOUT);
}

}  // namespace striped

using namespace striped;

extern "C" {

const char *striped_status_string(int status) {
    switch (status) {
        case STRIPED_OK: return "ok";
        case STRIPED_ERR_INVALID_ARG: return "invalid argument";
        case STRIPED_ERR_UNSUPPORTED: return "unsupported configuration";
        case STRIPED_ERR_ALIGN: return "misaligned pointer or stride";
        case STRIPED_ERR_CUDA: return "CUDA error";
        case STRIPED_ERR_TIMEOUT: return "device wait timed out";
        case STRIPED_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int striped_last_cuda_error(void) { return t_last_cuda_error; }

int striped_check_error(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e);
    int word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_status, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
    if (word != 0) {
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_status(e);
        return word;
    }
    return STRIPED_OK;
}

int striped_test_inject(int fault, int64_t wait_limit_ns) {
    if (fault < kInjectNone || fault > kInjectBwdSkipQ) return STRIPED_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();  // launches already queued keep their settings
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return STRIPED_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_state_mu);
    g_state[dev].limit_ns = wait_limit_ns > 0 ? (unsigned long long)wait_limit_ns : kDefaultWaitLimitNs;
    g_state[dev].inject = fault;
    return STRIPED_OK;
}

int striped_selftest_timeout(int64_t spins, void *stream) {
    if (spins < 0) return STRIPED_ERR_INVALID_ARG;
    selftest_wait_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(spins);
    return cuda_status(cudaGetLastError());
}

int striped_kernel_tile(int dtype, int64_t D, int *Tq, int *Tk) {
    if (!Tq || !Tk) return STRIPED_ERR_INVALID_ARG;
    if (dtype == STRIPED_BF16 && (D == 128 || D == 64)) {
        *Tq = *Tk = kTcTile;
        return STRIPED_OK;
    }
    if (dtype == STRIPED_FP32 && D % 8 == 0 && D <= 128 && D > 0) {
        *Tq = *Tk = kSimtTile;
        return STRIPED_OK;
    }
    return STRIPED_ERR_UNSUPPORTED;
}

int striped_fwd_query_tiles_per_cta(int64_t B, int64_t H, int64_t S, int64_t D, int N, int layout, int dtype,
                                    int num_sms) {
    const int st = check_attn(B, H, S, D, N, layout, dtype);
    if (st) return st;
    if (num_sms < 1) return STRIPED_ERR_INVALID_ARG;
    if (dtype != STRIPED_BF16) return 1;
    return fwd_pair_eligible(full_geom(B, H, H, S, D, N, layout, 1.0f), num_sms) ? 2 : 1;
}

// ---------------------------------------------------------------- permutation
// Packed sequences: check the HOST array cu_seqlens[0..nseq] (starts at 0,
// every length a positive multiple of N * unit rows) and build the table
// the kernels carry.  A length that is not a multiple of N (2N for zig-zag)
// has no placement (invalid); one that is, but not a whole number of `unit`
// rows per device, is a kernel restriction (unsupported).
static int make_seq_table(const int32_t *cu, int nseq, int N, int layout, int64_t unit, SeqTable *t,
                          int64_t *S) {
    if (!cu || nseq < 1 || N < 1) return STRIPED_ERR_INVALID_ARG;
    if (nseq > kMaxSeqs) return STRIPED_ERR_UNSUPPORTED;
    if (cu[0] != 0) return STRIPED_ERR_INVALID_ARG;
    const int64_t place = (layout == STRIPED_LAYOUT_ZIGZAG) ? 2 * (int64_t)N : (int64_t)N;
    int status = STRIPED_OK;
    for (int i = 0; i < nseq; ++i) {
        const int64_t len = (int64_t)cu[i + 1] - cu[i];
        if (len <= 0 || len % place != 0) return STRIPED_ERR_INVALID_ARG;
        if ((len / place) % unit != 0) status = STRIPED_ERR_UNSUPPORTED;
    }
    if (status != STRIPED_OK) return status;
    t->n = nseq;
    for (int i = 0; i <= nseq; ++i) t->row_start[i] = cu[i] / N;
    *S = cu[nseq];
    return STRIPED_OK;
}

static int permute_common(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                          int layout, int dtype, void *stream, bool gather, const SeqTable &seqs) {
    if (!x || !y) return STRIPED_ERR_INVALID_ARG;
    int st = check_sizes(B, H, S, D, N);
    if (st) return st;
    if (!valid_layout(layout)) return STRIPED_ERR_INVALID_ARG;
    if (layout == STRIPED_LAYOUT_ZIGZAG && S % (2 * (int64_t)N) != 0) return STRIPED_ERR_INVALID_ARG;
    int64_t esize;
    if (dtype == STRIPED_BF16) esize = 2;
    else if (dtype == STRIPED_FP32) esize = 4;
    else return STRIPED_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return STRIPED_ERR_ALIGN;
    if ((D * esize) % 16 != 0) return STRIPED_ERR_ALIGN;
    const char *xb = (const char *)x, *yb = (const char *)y;
    const int64_t bytes = B * H * S * D * esize;
    if (xb < yb + bytes && yb < xb + bytes) return STRIPED_ERR_INVALID_ARG;  // overlap
    return launch_stripe_permute(x, y, B * H, S, D * esize, N, layout, gather, seqs, (cudaStream_t)stream);
}

static const SeqTable kDense{};  // n = 0: one sequence per (batch, head)

int striped_permute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                    int dtype, void *stream) {
    return permute_common(x, y, B, H, S, D, N, STRIPED_LAYOUT_STRIPED, dtype, stream, true, kDense);
}

int striped_unpermute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                      int dtype, void *stream) {
    return permute_common(x, y, B, H, S, D, N, STRIPED_LAYOUT_STRIPED, dtype, stream, false, kDense);
}

int striped_layout_permute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                           int layout, int dtype, void *stream) {
    return permute_common(x, y, B, H, S, D, N, layout, dtype, stream, true, kDense);
}

int striped_layout_unpermute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D,
                             int N, int layout, int dtype, void *stream) {
    return permute_common(x, y, B, H, S, D, N, layout, dtype, stream, false, kDense);
}

int striped_varlen_permute(const void *x, void *y, const int32_t *cu_seqlens, int nseq, int64_t H, int64_t D,
                           int N, int layout, int dtype, void *stream) {
    SeqTable t{};
    int64_t S = 0;
    const int st = make_seq_table(cu_seqlens, nseq, N, layout, 1, &t, &S);
    if (st) return st;
    return permute_common(x, y, 1, H, S, D, N, layout, dtype, stream, true, t);
}

int striped_varlen_unpermute(const void *x, void *y, const int32_t *cu_seqlens, int nseq, int64_t H, int64_t D,
                             int N, int layout, int dtype, void *stream) {
    SeqTable t{};
    int64_t S = 0;
    const int st = make_seq_table(cu_seqlens, nseq, N, layout, 1, &t, &S);
    if (st) return st;
    return permute_common(x, y, 1, H, S, D, N, layout, dtype, stream, false, t);
}

// ---------------------------------------------------------------- attention
static int check_heads(int64_t H, int64_t Hkv) {
    return (Hkv >= 1 && Hkv <= H && H % Hkv == 0) ? STRIPED_OK : STRIPED_ERR_INVALID_ARG;
}

int striped_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, int N, int layout, int dtype, float scale,
                     int64_t *tile_stats, void *stream) {
    return striped_attn_fwd_gqa(q, k, v, o, lse, B, H, H, S, D, N, layout, dtype, scale, tile_stats, stream);
}

static int attn_fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                           int64_t H, int64_t Hkv, int64_t S, int64_t D, int N, int layout, int dtype,
                           float scale, int64_t *tile_stats, void *stream, const SeqTable &seqs) {
    if (!q || !k || !v || !o || !lse) return STRIPED_ERR_INVALID_ARG;
    int st = check_attn(B, H, S, D, N, layout, dtype);
    if (st) return st;
    if ((st = check_heads(H, Hkv))) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return STRIPED_ERR_ALIGN;
    AttnGeom g = full_geom(B, H, Hkv, S, D, N, layout, scale);
    g.seqs = seqs;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == STRIPED_FP32)
        return launch_simt_fwd((const float *)q, (const float *)k, (const float *)v, (float *)o, lse, g,
                               tile_stats, s);
    return launch_tc_fwd(q, k, v, o, lse, g, tile_stats, s);
}

int striped_attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                         int64_t H, int64_t Hkv, int64_t S, int64_t D, int N, int layout, int dtype,
                         float scale, int64_t *tile_stats, void *stream) {
    return attn_fwd_common(q, k, v, o, lse, B, H, Hkv, S, D, N, layout, dtype, scale, tile_stats, stream, kDense);
}

// the kernel tile for dtype (128 for bf16 tensor cores, 16 for fp32)
static int64_t tile_of(int dtype) { return dtype == STRIPED_BF16 ? kTcTile : kSimtTile; }

int striped_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int32_t *cu_seqlens, int nseq, int64_t H, int64_t Hkv, int64_t D, int N,
                            int layout, int dtype, float scale, int64_t *tile_stats, void *stream) {
    SeqTable t{};
    int64_t S = 0;
    const int st = make_seq_table(cu_seqlens, nseq, N, layout, tile_of(dtype), &t, &S);
    if (st) return st;
    return attn_fwd_common(q, k, v, o, lse, 1, H, Hkv, S, D, N, layout, dtype, scale, tile_stats, stream, t);
}

// bf16 workspace: fp32 dQ accumulator [B*H*S][D], then per (b, h, stripe)
// and 128-row tile a statistics block [LSE*log2e 128 | Delta 128] (fp32).
static size_t bf16_stats_offset(int64_t B, int64_t H, int64_t S, int64_t D) {
    return align256((size_t)(B * H * S) * (size_t)D * sizeof(float));
}

size_t striped_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D, int N, int dtype) {
    if (B < 1 || H < 1 || S < 1 || D < 1 || N < 1 || S % N != 0) return 0;
    const size_t rows = (size_t)(B * H * S);
    if (dtype == STRIPED_FP32) return align256(rows * sizeof(float));
    if (dtype == STRIPED_BF16) {
        const size_t nq = (size_t)((S / N + kTcTile - 1) / kTcTile);
        return bf16_stats_offset(B, H, S, D) + align256((size_t)(B * H * N) * nq * 2 * kTcTile * sizeof(float));
    }
    return 0;
}

int striped_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dO, void *dq, void *dk, void *dv, void *workspace,
                     size_t ws_bytes, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                     int layout, int dtype, float scale, int64_t *tile_stats, void *stream) {
    return striped_attn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, B, H, H, S, D, N, layout,
                                dtype, scale, tile_stats, stream);
}

static int attn_bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
                           const void *dO, void *dq, void *dk, void *dv, void *workspace, size_t ws_bytes,
                           int64_t B, int64_t H, int64_t Hkv, int64_t S, int64_t D, int N, int layout,
                           int dtype, float scale, int64_t *tile_stats, void *stream, const SeqTable &seqs) {
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return STRIPED_ERR_INVALID_ARG;
    int st = check_attn(B, H, S, D, N, layout, dtype);
    if (st) return st;
    if ((st = check_heads(H, Hkv))) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return STRIPED_ERR_ALIGN;
    const size_t need = striped_workspace_size(B, H, S, D, N, dtype);
    if (!workspace || ws_bytes < need) return STRIPED_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return STRIPED_ERR_ALIGN;
    AttnGeom g = full_geom(B, H, Hkv, S, D, N, layout, scale);
    g.seqs = seqs;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == STRIPED_FP32)
        return launch_simt_bwd((const float *)q, (const float *)k, (const float *)v, (const float *)o, lse,
                               (const float *)dO, (float *)dq, (float *)dk, (float *)dv,
                               (float *)workspace, g, tile_stats, s);
    float *dq_acc = (float *)workspace;
    float *stats = (float *)((char *)workspace + bf16_stats_offset(B, H, S, D));
    return launch_tc_bwd(q, k, v, o, lse, dO, dq, dk, dv, dq_acc, stats, g, tile_stats, s);
}

int striped_attn_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dO, void *dq, void *dk, void *dv, void *workspace,
                         size_t ws_bytes, int64_t B, int64_t H, int64_t Hkv, int64_t S, int64_t D, int N,
                         int layout, int dtype, float scale, int64_t *tile_stats, void *stream) {
    return attn_bwd_common(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, B, H, Hkv, S, D, N, layout,
                           dtype, scale, tile_stats, stream, kDense);
}

int striped_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                            const void *dO, void *dq, void *dk, void *dv, void *workspace, size_t ws_bytes,
                            const int32_t *cu_seqlens, int nseq, int64_t H, int64_t Hkv, int64_t D, int N,
                            int layout, int dtype, float scale, int64_t *tile_stats, void *stream) {
    SeqTable t{};
    int64_t S = 0;
    const int st = make_seq_table(cu_seqlens, nseq, N, layout, tile_of(dtype), &t, &S);
    if (st) return st;
    return attn_bwd_common(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, 1, H, Hkv, S, D, N, layout,
                           dtype, scale, tile_stats, stream, t);
}

size_t ring_bwd_workspace_size(int64_t B, int64_t H, int64_t L, int64_t D, int dtype) {
    if (B < 1 || H < 1 || L < 1 || D < 1 || dtype != STRIPED_BF16) return 0;
    const size_t nq = (size_t)((L + kTcTile - 1) / kTcTile);
    return align256((size_t)(B * H) * nq * 2 * kTcTile * sizeof(float));
}

// the geometry of one device's blocks: contiguous [BH][L][D], no stripes
static AttnGeom round_geom(int64_t B, int64_t H, int64_t L, int64_t D, int N, int layout, float scale) {
    AttnGeom g{};
    g.BH = B * H;
    g.G = 1;
    g.L = L;
    g.D = D;
    g.N = N;
    g.layout = layout;
    g.stride_bh = L * D;
    g.stripe_stride = 0;
    g.lse_stride_bh = L;
    g.lse_stripe_stride = 0;
    g.scale = scale;
    return g;
}

int ring_bwd_prepare(const void *o_d, const float *lse_d, const void *dO_d, void *workspace, size_t ws_bytes,
                     float *dq_acc_d, int64_t B, int64_t H, int64_t L, int64_t D, int dtype, void *stream) {
    if (!o_d || !lse_d || !dO_d || !dq_acc_d) return STRIPED_ERR_INVALID_ARG;
    int st = check_sizes(B, H, L, D, 1);
    if (st) return st;
    if (dtype == STRIPED_FP32) return STRIPED_ERR_UNSUPPORTED;
    if (dtype != STRIPED_BF16) return STRIPED_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return STRIPED_ERR_UNSUPPORTED;
    if (!aligned16(o_d) || !aligned16(dO_d) || !aligned16(dq_acc_d)) return STRIPED_ERR_ALIGN;
    if (!workspace || ws_bytes < ring_bwd_workspace_size(B, H, L, D, dtype)) return STRIPED_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return STRIPED_ERR_ALIGN;
    return launch_round_bwd_prepare(o_d, lse_d, dO_d, (float *)workspace, dq_acc_d,
                                    round_geom(B, H, L, D, 1, STRIPED_LAYOUT_STRIPED, 1.f), (cudaStream_t)stream);
}

int ring_round_bwd(const void *q_d, const void *k_e, const void *v_e, const void *dO_d, const void *workspace,
                   size_t ws_bytes, float *dq_acc_d, float *dk_acc_e, float *dv_acc_e, int d, int e, int64_t B,
                   int64_t H, int64_t L, int64_t D, int N, int layout, int dtype, float scale, int first_round,
                   int64_t *tile_stats, void *stream) {
    if (!q_d || !k_e || !v_e || !dO_d || !dq_acc_d || !dk_acc_e || !dv_acc_e) return STRIPED_ERR_INVALID_ARG;
    if (L < 1) return STRIPED_ERR_INVALID_ARG;
    int st = check_attn(B, H, L * N, D, N, layout, dtype);
    if (st) return st;
    if (dtype == STRIPED_FP32) return STRIPED_ERR_UNSUPPORTED;
    if (d < 0 || d >= N || e < 0 || e >= N) return STRIPED_ERR_INVALID_ARG;
    if (!aligned16(q_d) || !aligned16(k_e) || !aligned16(v_e) || !aligned16(dO_d) || !aligned16(dq_acc_d) ||
        !aligned16(dk_acc_e) || !aligned16(dv_acc_e))
        return STRIPED_ERR_ALIGN;
    if (!workspace || ws_bytes < ring_bwd_workspace_size(B, H, L, D, dtype)) return STRIPED_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return STRIPED_ERR_ALIGN;
    return launch_tc_round_bwd(q_d, k_e, v_e, dO_d, (const float *)workspace, dq_acc_d, dk_acc_e, dv_acc_e, d, e,
                               first_round ? 1 : 0, round_geom(B, H, L, D, N, layout, scale), tile_stats,
                               (cudaStream_t)stream);
}

int ring_bwd_finish(const float *acc, void *out, int64_t n, int dtype, float mul, void *stream) {
    if (!acc || !out || n < 0 || n % 8 != 0) return STRIPED_ERR_INVALID_ARG;
    if (dtype == STRIPED_FP32) return STRIPED_ERR_UNSUPPORTED;
    if (dtype != STRIPED_BF16) return STRIPED_ERR_INVALID_ARG;
    if (!aligned16(acc) || !aligned16(out)) return STRIPED_ERR_ALIGN;
    if (n == 0) return STRIPED_OK;
    return launch_scale_to_bf16(acc, out, n / 8, mul, (cudaStream_t)stream);
}

int ring_round_fwd(const void *q_d, const void *k_e, const void *v_e, float *o_acc, float *lse_acc,
                   void *o_out, int d, int e, int64_t B, int64_t H, int64_t L, int64_t D, int N,
                   int64_t stride_bh, int64_t lse_stride_bh, int layout, int dtype, float scale,
                   int first_round, int64_t *tile_stats, void *stream) {
    if (!q_d || !k_e || !v_e || !o_acc || !lse_acc) return STRIPED_ERR_INVALID_ARG;
    if (L < 1) return STRIPED_ERR_INVALID_ARG;
    int st = check_attn(B, H, L * N, D, N, layout, dtype);
    if (st) return st;
    if (d < 0 || d >= N || e < 0 || e >= N) return STRIPED_ERR_INVALID_ARG;
    if (stride_bh < L * D || lse_stride_bh < L) return STRIPED_ERR_INVALID_ARG;
    if (!aligned16(q_d) || !aligned16(k_e) || !aligned16(v_e) || !aligned16(o_acc) ||
        (o_out && !aligned16(o_out)))
        return STRIPED_ERR_ALIGN;
    const int64_t esize = dtype == STRIPED_BF16 ? 2 : 4;
    if ((stride_bh * esize) % 16 != 0 || (stride_bh * 4) % 16 != 0) return STRIPED_ERR_ALIGN;
    AttnGeom g{};  // seqs.n = 0: dense
    g.BH = B * H;
    g.G = 1;
    g.L = L;
    g.D = D;
    g.N = N;
    g.layout = layout;
    g.stride_bh = stride_bh;
    g.stripe_stride = 0;
    g.lse_stride_bh = lse_stride_bh;
    g.lse_stripe_stride = 0;
    g.scale = scale;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == STRIPED_FP32)
        return launch_simt_round((const float *)q_d, (const float *)k_e, (const float *)v_e, o_acc, lse_acc,
                                 (float *)o_out, d, e, first_round ? 1 : 0, g, tile_stats, s);
    return launch_tc_round(q_d, k_e, v_e, o_acc, lse_acc, o_out, d, e, first_round ? 1 : 0, g, tile_stats,
                           s);
}

}  // extern "C"
