// permute.cu -- stripe permutation of [B, H, S, D] tensors (HBM-bound copy).
//
// Striped Attention gives virtual device d every N-th token: positions
// p = i*N + d, i < L = S/N ("every N-th token", research.elamur.ai summary
// page, §Summary), applied once before the model (§Key points "Striped
// layout").  Stripe-major row d*L + i therefore holds position i*N + d.
//
//   permute   (gather):  y[d*L + i] = x[i*N + d]
//   unpermute (scatter): y[i*N + d] = x[d*L + i]
//
// The same kernel serves the other row orders with their own row -> position
// map: contiguous (position d*L + i, a copy) and zig-zag (device d holds
// chunk d then chunk 2N-1-d of 2N chunks of C = L/2 positions), and packed
// variable-length batches, where each sequence is placed on its own and a
// device's slice holds its rows of every sequence in turn.
//
// One block moves a run of consecutive stripe rows of one (b, h) head; the
// stripe index d is uniform per block (no per-element division).  Each row
// is D*esize bytes moved as 16-byte vectors (vpr of them; a power of two
// takes shifts and masks, any other count a division); a thread issues all
// its loads before its stores so that every thread keeps several requests
// in flight.
#include "common.cuh"
#include "internal.h"

namespace striped {

constexpr int kPermThreads = 256;
constexpr int kPermVecPerThread = 8;  // 16-byte vectors per thread per block

// Position of row i of device d under the placement kLayout.
template <int kLayout>
__device__ __forceinline__ int64_t position_of(int64_t d, int64_t i, int64_t L, int N) {
    if (kLayout == STRIPED_LAYOUT_CONTIGUOUS) return d * L + i;
    if (kLayout == STRIPED_LAYOUT_ZIGZAG) {
        const int64_t C = L >> 1;
        return i < C ? d * C + i : (2 * (int64_t)N - 1 - d) * C + (i - C);
    }
    return i * N + d;
}

// Position of row i of device d's slice in a packed head: the row's
// sequence (its first row sq.start in the slice, sq.count rows per device)
// starts at position sq.start * N.
template <int kLayout>
__device__ __forceinline__ int64_t packed_position_of(const SeqTable &seqs, int64_t d, int64_t i, int64_t L, int N) {
    if (seqs.n == 0) return position_of<kLayout>(d, i, L, N);
    const SeqSpan sq = seq_of(seqs, (int)i, 1, (int)L);
    return (int64_t)sq.start * N + position_of<kLayout>(d, i - sq.start, sq.count, N);
}

template <int kLayout, bool kGather, bool kPow2>
__global__ void __launch_bounds__(kPermThreads) stripe_permute_kernel(
    const uint4 *__restrict__ x, uint4 *__restrict__ y, int64_t S, int64_t L, int N, int vpr_arg,
    int vec_per_row_log2, int rows_per_block, int blocks_per_stripe, const __grid_constant__ SeqTable seqs) {
    const int64_t bh = blockIdx.y;
    const int d = blockIdx.x / blocks_per_stripe;
    const int64_t i0 = (int64_t)(blockIdx.x % blocks_per_stripe) * rows_per_block;
    const int vpr = kPow2 ? 1 << vec_per_row_log2 : vpr_arg;
    const int64_t head = bh * S;  // row offset of this head
    const int nvec = rows_per_block * vpr;

    uint4 buf[kPermVecPerThread];
    int64_t dst_idx[kPermVecPerThread];
#pragma unroll
    for (int u = 0; u < kPermVecPerThread; ++u) {
        const int v = threadIdx.x + u * kPermThreads;
        dst_idx[u] = -1;
        if (v < nvec) {
            const int r = kPow2 ? v >> vec_per_row_log2 : v / vpr;
            const int64_t i = i0 + r;
            const int c = kPow2 ? v & (vpr - 1) : v - r * vpr;
            if (i < L) {
                const int64_t striped_row = head + (int64_t)d * L + i;
                const int64_t pos_row = head + packed_position_of<kLayout>(seqs, d, i, L, N);
                const int64_t src = (kGather ? pos_row : striped_row) * vpr + c;
                dst_idx[u] = (kGather ? striped_row : pos_row) * vpr + c;
                buf[u] = __ldg(x + src);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kPermVecPerThread; ++u)
        if (dst_idx[u] >= 0) y[dst_idx[u]] = buf[u];
}

template <int kLayout, bool kPow2>
static void launch_layout2(dim3 grid, cudaStream_t stream, bool gather, const void *x, void *y, int64_t S,
                           int64_t L, int N, int vpr, int vlog, int rows_per_block, int bps, const SeqTable &seqs) {
    if (gather)
        stripe_permute_kernel<kLayout, true, kPow2><<<grid, kPermThreads, 0, stream>>>(
            (const uint4 *)x, (uint4 *)y, S, L, N, vpr, vlog, rows_per_block, bps, seqs);
    else
        stripe_permute_kernel<kLayout, false, kPow2><<<grid, kPermThreads, 0, stream>>>(
            (const uint4 *)x, (uint4 *)y, S, L, N, vpr, vlog, rows_per_block, bps, seqs);
}

template <int kLayout>
static void launch_layout(dim3 grid, cudaStream_t stream, bool gather, const void *x, void *y, int64_t S,
                          int64_t L, int N, int vpr, int vlog, int rows_per_block, int bps, const SeqTable &seqs) {
    if ((1 << vlog) == vpr)
        launch_layout2<kLayout, true>(grid, stream, gather, x, y, S, L, N, vpr, vlog, rows_per_block, bps, seqs);
    else
        launch_layout2<kLayout, false>(grid, stream, gather, x, y, S, L, N, vpr, vlog, rows_per_block, bps, seqs);
}

int launch_stripe_permute(const void *x, void *y, int64_t BH, int64_t S, int64_t row_bytes, int N,
                          int layout, bool gather, const SeqTable &seqs, cudaStream_t stream) {
    const int64_t L = S / N;
    if (row_bytes < 16 || row_bytes % 16 != 0) return STRIPED_ERR_UNSUPPORTED;
    const int64_t vpr = row_bytes / 16;
    if (vpr > kPermThreads * kPermVecPerThread) return STRIPED_ERR_UNSUPPORTED;
    int vlog = 0;
    while ((1ll << vlog) < vpr) ++vlog;
    // rows per block such that the block moves at most kPermThreads*kPermVecPerThread vectors
    const int rows_per_block = (int)((kPermThreads * kPermVecPerThread) / vpr);
    const int64_t bps = (L + rows_per_block - 1) / rows_per_block;
    if (bps * N > 0x7fffffffll || BH > 65535) return STRIPED_ERR_UNSUPPORTED;
    dim3 grid((unsigned)(bps * N), (unsigned)BH);
    if (layout == STRIPED_LAYOUT_ZIGZAG)
        launch_layout<STRIPED_LAYOUT_ZIGZAG>(grid, stream, gather, x, y, S, L, N, (int)vpr, vlog, rows_per_block,
                                             (int)bps, seqs);
    else if (layout == STRIPED_LAYOUT_CONTIGUOUS)
        launch_layout<STRIPED_LAYOUT_CONTIGUOUS>(grid, stream, gather, x, y, S, L, N, (int)vpr, vlog, rows_per_block,
                                                 (int)bps, seqs);
    else
        launch_layout<STRIPED_LAYOUT_STRIPED>(grid, stream, gather, x, y, S, L, N, (int)vpr, vlog, rows_per_block,
                                              (int)bps, seqs);
    return cuda_status(cudaGetLastError());
}

}  // namespace striped
