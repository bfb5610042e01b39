// attn_simt.cu -- fp32 striped causal attention on the CUDA cores.
//
// The fp32 path keeps every product in fp32 (TF32 tensor cores would round
// the operands to 10 mantissa bits).  Same method and schedule as the
// tensor-core path: the query tile of virtual device d visits, in ring
// rounds r = 0..N-1, the key stripe e = (d - r) mod N (research.elamur.ai
// summary page, §Summary); fully masked tiles are skipped; the rounds are
// merged by an online softmax, so the result is exact causal attention
// (pith.science paper page, abstract).
//
// Block = kSimtTile query (or key) rows x 8 threads per row; each thread
// owns D/8 of the head dimension and dot products are reduced over the 8
// threads of a row with warp shuffles.  Key/value (or query/dO) tiles are
// staged in shared memory; the 16 scores of a tile are formed together (so
// their dot products, shuffles and exponentials overlap) and the forward's
// running maximum is updated once per tile.  The kernels are instantiated
// for D/8 = 8 and 16 (D = 64, 128) and, for the other multiples of 8, with
// D/8 read at run time.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace striped {

namespace {

constexpr int T = kSimtTile;
constexpr int kTPR = 8;             // threads per row
constexpr int kThreads = T * kTPR;  // 128
constexpr int kMaxDPT = 16;         // D <= 128
// keys (query rows) per chunk in the gradient kernels: the unrolled chunk
// keeps its K/Q and V/dO rows in flight, so it shrinks as D grows
template <int DPT>
__host__ __device__ constexpr int grad_chunk() { return DPT == 16 ? 4 : 8; }

__device__ __forceinline__ float group_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

__device__ __forceinline__ int rows_in_tile(int64_t L, int t) {
    const int64_t r = L - (int64_t)t * T;
    return r >= T ? T : (int)r;
}

// Head dimension of an instantiation: DPT = D/8 elements per thread, or 0
// for D read at run time.
template <int DPT>
struct Dim {
    static constexpr int kU = DPT ? DPT : kMaxDPT;  // unrolled loop bound
    int dpt, D;
    __device__ __forceinline__ explicit Dim(int64_t d) : dpt(DPT ? DPT : (int)d / kTPR), D(DPT ? DPT * kTPR : (int)d) {}
};

// One thread's share of tile t of a stripe (T rows of D floats, zero
// beyond L) as 16-byte vectors (D is a multiple of 8): loaded into
// registers while the previous tile is computed, then stored to shared
// memory.
constexpr int kMaxF4 = (T * kMaxDPT * kTPR / 4 + kThreads - 1) / kThreads;  // 4
template <int DPT>
struct TileRegs {
    static constexpr int kN = DPT ? (T * DPT * kTPR / 4 + kThreads - 1) / kThreads : kMaxF4;
    float4 v[kN];
};

template <int DPT>
__device__ __forceinline__ void tile_load(TileRegs<DPT> &r, const float *src_stripe, int64_t L, const Dim<DPT> &dm,
                                          int t) {
    const int rows = rows_in_tile(L, t);
    const int D4 = dm.D / 4;
    const float4 *src = reinterpret_cast<const float4 *>(src_stripe + (int64_t)t * T * dm.D);
#pragma unroll
    for (int k = 0; k < TileRegs<DPT>::kN; ++k) {
        const int idx = threadIdx.x + k * kThreads;
        r.v[k] = (idx < T * D4 && idx / D4 < rows) ? src[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int DPT>
__device__ __forceinline__ void tile_store(const TileRegs<DPT> &r, float *dst, const Dim<DPT> &dm) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int k = 0; k < TileRegs<DPT>::kN; ++k) {
        const int idx = threadIdx.x + k * kThreads;
        if (idx < T * (dm.D / 4)) d4[idx] = r.v[k];
    }
}

struct RowState {
    float m, l;
    float acc[kMaxDPT];
};

// Online-softmax forward of query tile ag of stripe d over rounds
// [r_lo, r_hi) (e_fixed >= 0: the single key stripe e_fixed).  With packed
// sequences the schedule runs over the tiles of ag's own sequence.
template <int DPT>
__device__ void fwd_tile(const float *__restrict__ q_stripe, const float *__restrict__ k_head,
                         const float *__restrict__ v_head, const AttnGeom &g, int d, int ag, int r_lo,
                         int r_hi, int e_fixed, RowState &st, int64_t *tile_stats, float *sK,
                         float *sV) {
    constexpr int kU = Dim<DPT>::kU;
    const Dim<DPT> dm(g.D);
    const int64_t L = g.L;
    const int D = dm.D, dpt = dm.dpt;
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
    const int nq = (int)((L + T - 1) / T);
    const int rows_a = rows_in_tile(L, ag);
    const int64_t i = (int64_t)ag * T + row;
    const SeqSpan sq = seq_of(g.seqs, ag, T, nq);
    const int a = ag - sq.start, nqs = sq.count;
    float qreg[kU];
#pragma unroll
    for (int c = 0; c < kU; ++c)
        qreg[c] = (c < dpt && i < L) ? q_stripe[i * D + sub * dpt + c] : 0.f;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxDPT; ++c) st.acc[c] = 0.f;

    // the (round, key tile) sequence of this query tile; the next tile's K
    // and V are loaded into registers while the current one is computed
    struct Cur {
        int r, b, e, ntiles;
        RoundSpan sp;
    };
    auto seek = [&](Cur &c) -> bool {
        for (; c.r < r_hi; ++c.r, c.b = 0) {
            c.e = e_fixed >= 0 ? e_fixed : (d - c.r + g.N) % g.N;
            c.sp = round_span(g.layout, d, c.e, a, nqs, rows_a);
            c.ntiles = c.sp.nfull + c.sp.has_diag;
            if (c.b < c.ntiles) return true;
        }
        return false;
    };
    Cur cur{r_lo, 0, 0, 0, RoundSpan{0, 0, 0}};
    bool have = seek(cur);
    TileRegs<DPT> rk, rv;
    if (have) {
        tile_load(rk, k_head + (int64_t)cur.e * g.stripe_stride, L, dm, sq.start + cur.b);
        tile_load(rv, v_head + (int64_t)cur.e * g.stripe_stride, L, dm, sq.start + cur.b);
    }
    // tiles of the current round processed so far (full / partial), added to
    // the round's counters when the round ends
    int n_full = 0, n_part = 0;
    while (have) {
        __syncthreads();
        tile_store(rk, sK, dm);
        tile_store(rv, sV, dm);
        __syncthreads();
        Cur nxt = cur;
        ++nxt.b;
        const bool have_next = seek(nxt);
        if (have_next) {
            tile_load(rk, k_head + (int64_t)nxt.e * g.stripe_stride, L, dm, sq.start + nxt.b);
            tile_load(rv, v_head + (int64_t)nxt.e * g.stripe_stride, L, dm, sq.start + nxt.b);
        }
        const RoundSpan &sp = cur.sp;
        const int b = cur.b;
        {
            const int rows_b = rows_in_tile(L, sq.start + b);
            const bool diag = sp.has_diag && b == sp.nfull;
            // the tile's scores; rows past the stripe end and masked pairs
            // become -inf and drop out of the max and the sums
            float sc[T];
#pragma unroll
            for (int c = 0; c < T; ++c) {
                float part = 0.f;
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (u < dpt) part += qreg[u] * sK[c * D + sub * dpt + u];
                sc[c] = part;
            }
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < T; ++c) {
                const float s = g.scale * group_sum(sc[c]);
                const bool keep = c < rows_b && (!diag || c <= row + sp.diag_off);
                sc[c] = keep ? s : -INFINITY;
                mt = fmaxf(mt, sc[c]);
            }
            if (mt != -INFINITY) {
                const float m_new = fmaxf(st.m, mt);
                const float alpha = expf(st.m - m_new);  // exp(-inf) = 0 on the first kept key
                float lsum = 0.f;
#pragma unroll
                for (int c = 0; c < T; ++c) {
                    sc[c] = expf(sc[c] - m_new);
                    lsum += sc[c];
                }
                st.l = st.l * alpha + lsum;
#pragma unroll
                for (int u = 0; u < kU; ++u) st.acc[u] *= alpha;
#pragma unroll
                for (int c = 0; c < T; ++c)
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (u < dpt) st.acc[u] += sc[c] * sV[c * D + sub * dpt + u];
                st.m = m_new;
            }
            if (diag) ++n_part;
            else ++n_full;
        }
        if (!have_next || nxt.r != cur.r) {
            if (tile_stats && threadIdx.x == 0) {
                const int rr = ring_round_of(d, cur.e, g.N);
                atomicAdd((unsigned long long *)&tile_stats[rr * g.N + d], (unsigned long long)n_full);
                atomicAdd((unsigned long long *)&tile_stats[g.N * g.N + rr * g.N + d], (unsigned long long)n_part);
            }
            n_full = n_part = 0;
        }
        cur = nxt;
        have = have_next;
    }
}

template <int DPT>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(const float *__restrict__ q,
                                                             const float *__restrict__ k,
                                                             const float *__restrict__ v,
                                                             float *__restrict__ o,
                                                             float *__restrict__ lse, AttnGeom g,
                                                             int64_t *tile_stats) {
    extern __shared__ __align__(16) float smem[];
    float *sK = smem, *sV = smem + T * g.D;
    const int nq = (int)((g.L + T - 1) / T);
    const int a = nq - 1 - (int)(blockIdx.x % nq);  // heavy query tiles first
    const int d = (int)(blockIdx.x / nq);
    const int64_t bh = blockIdx.y;
    const int64_t kvh = bh / g.G;  // key/value head of query head bh
    const float *q_stripe = q + bh * g.stride_bh + (int64_t)d * g.stripe_stride;
    RowState st;
    fwd_tile<DPT>(q_stripe, k + kvh * g.stride_bh, v + kvh * g.stride_bh, g, d, a, 0, g.N, -1, st,
                  tile_stats, sK, sV);
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
    const int64_t i = (int64_t)a * T + row;
    if (i >= g.L) return;
    const int dpt = Dim<DPT>(g.D).dpt;
    float *orow = o + bh * g.stride_bh + (int64_t)d * g.stripe_stride + i * g.D + sub * dpt;
    const float inv = 1.f / st.l;
#pragma unroll
    for (int u = 0; u < Dim<DPT>::kU; ++u)
        if (u < dpt) orow[u] = st.acc[u] * inv;
    if (sub == 0)
        lse[bh * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride + i] = st.m + logf(st.l);
}

template <int DPT>
__global__ void __launch_bounds__(kThreads) simt_round_kernel(
    const float *__restrict__ q_d, const float *__restrict__ k_e, const float *__restrict__ v_e,
    float *__restrict__ o_acc, float *__restrict__ lse_acc, float *__restrict__ o_out, int d, int e,
    int first, AttnGeom g, int64_t *tile_stats) {
    extern __shared__ __align__(16) float smem[];
    float *sK = smem, *sV = smem + T * g.D;
    const int nq = (int)((g.L + T - 1) / T);
    const int a = nq - 1 - (int)blockIdx.x;
    const int64_t bh = blockIdx.y;
    RowState st;
    // the launcher sets stripe_stride = 0: k_e / v_e are the stripe slices
    fwd_tile<DPT>(q_d + bh * g.stride_bh, k_e + bh * g.stride_bh, v_e + bh * g.stride_bh, g, d, a, 0, 1,
                  e, st, tile_stats, sK, sV);
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
    const int64_t i = (int64_t)a * T + row;
    if (i >= g.L) return;
    const int dpt = Dim<DPT>(g.D).dpt;
    // this round's normalised partial result; LSE_r = -inf when nothing kept
    const bool empty = !(st.l > 0.f);
    const float lse_r = empty ? -INFINITY : st.m + logf(st.l);
    float *acc_row = o_acc + bh * g.stride_bh + i * g.D + sub * dpt;
    float *lse_ptr = lse_acc + bh * g.lse_stride_bh + i;
    const float lse_a = first ? -INFINITY : *lse_ptr;
    const float mx = fmaxf(lse_a, lse_r);
    float wa = 0.f, wr = 0.f, lse_new = -INFINITY;
    if (mx != -INFINITY) {
        wa = expf(lse_a - mx);
        wr = expf(lse_r - mx);
        lse_new = mx + logf(wa + wr);
        const float inv = 1.f / (wa + wr);
        wa *= inv;
        wr *= inv;
    }
    const float inv_l = empty ? 0.f : 1.f / st.l;
#pragma unroll
    for (int u = 0; u < Dim<DPT>::kU; ++u) {
        if (u >= dpt) continue;
        const float o_r = st.acc[u] * inv_l;
        float val;
        if (mx == -INFINITY) val = first ? 0.f : acc_row[u];
        else val = (first ? 0.f : wa * acc_row[u]) + wr * o_r;
        acc_row[u] = val;
        if (o_out) o_out[bh * g.stride_bh + i * g.D + sub * dpt + u] = val;
    }
    __syncwarp();
    if (sub == 0) *lse_ptr = lse_new;
}

// Delta_p = <dO_p, O_p>: one warp per row.
__global__ void simt_delta_kernel(const float *__restrict__ o, const float *__restrict__ dO,
                                  float *__restrict__ delta, int64_t rows, int64_t D) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= rows) return;
    float s = 0.f;
    for (int64_t c = lane; c < D; c += 32) s += o[row * D + c] * dO[row * D + c];
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) delta[row] = s;
}

// dQ: query tile of stripe d, same schedule as the forward.
template <int DPT>
__global__ void __launch_bounds__(kThreads) simt_dq_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ lse, const float *__restrict__ dO, const float *__restrict__ delta,
    float *__restrict__ dq, AttnGeom g, int64_t *tile_stats) {
    extern __shared__ __align__(16) float smem[];
    float *sK = smem, *sV = smem + T * g.D;
    constexpr int kU = Dim<DPT>::kU, kCh = grad_chunk<DPT>();
    const Dim<DPT> dm(g.D);
    const int64_t L = g.L;
    const int D = dm.D, dpt = dm.dpt;
    const int nq = (int)((L + T - 1) / T);
    const int ag = nq - 1 - (int)(blockIdx.x % nq);
    const int d = (int)(blockIdx.x / nq);
    const int64_t bh = blockIdx.y;
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;
    const int64_t i = (int64_t)ag * T + row;
    const bool valid = i < L;
    const SeqSpan sq = seq_of(g.seqs, ag, T, nq);  // packed sequences: own sequence's tiles
    const int a = ag - sq.start, nqs = sq.count;
    const int64_t qoff = bh * g.stride_bh + (int64_t)d * g.stripe_stride + i * D + sub * dpt;
    const int64_t soff = bh * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride + i;
    float qreg[kU], doreg[kU], acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        qreg[u] = (u < dpt && valid) ? q[qoff + u] : 0.f;
        doreg[u] = (u < dpt && valid) ? dO[qoff + u] : 0.f;
        acc[u] = 0.f;
    }
    const float lse_i = valid ? lse[soff] : 0.f;
    const float delta_i = valid ? delta[soff] : 0.f;
    const int rows_a = rows_in_tile(L, ag);
    const float *k_head = k + (bh / g.G) * g.stride_bh, *v_head = v + (bh / g.G) * g.stride_bh;
    // the (round, key tile) sequence, the next tile loading during this one
    struct Cur {
        int r, b, e, ntiles;
        RoundSpan sp;
    };
    auto seek = [&](Cur &c) -> bool {
        for (; c.r < g.N; ++c.r, c.b = 0) {
            c.e = (d - c.r + g.N) % g.N;
            c.sp = round_span(g.layout, d, c.e, a, nqs, rows_a);
            c.ntiles = c.sp.nfull + c.sp.has_diag;
            if (c.b < c.ntiles) return true;
        }
        return false;
    };
    Cur cur{0, 0, 0, 0, RoundSpan{0, 0, 0}};
    bool have = seek(cur);
    TileRegs<DPT> rk, rv;
    if (have) {
        tile_load(rk, k_head + (int64_t)cur.e * g.stripe_stride, L, dm, sq.start + cur.b);
        tile_load(rv, v_head + (int64_t)cur.e * g.stripe_stride, L, dm, sq.start + cur.b);
    }
    int n_full = 0, n_part = 0;  // tiles of the current round, counted as they run
    while (have) {
        __syncthreads();
        tile_store(rk, sK, dm);
        tile_store(rv, sV, dm);
        __syncthreads();
        Cur nxt = cur;
        ++nxt.b;
        const bool have_next = seek(nxt);
        if (have_next) {
            tile_load(rk, k_head + (int64_t)nxt.e * g.stripe_stride, L, dm, sq.start + nxt.b);
            tile_load(rv, v_head + (int64_t)nxt.e * g.stripe_stride, L, dm, sq.start + nxt.b);
        }
        const RoundSpan &sp = cur.sp;
        {
            const int b = cur.b;
            const int rows_b = rows_in_tile(L, sq.start + b);
            const bool diag = sp.has_diag && b == sp.nfull;
            // the tile's keys in chunks of kCh (a rolled loop bounds the
            // registers the unrolled chunk keeps live)
#pragma unroll 1
            for (int c0 = 0; c0 < T; c0 += kCh) {
                float ps[kCh], pp[kCh];
#pragma unroll
                for (int c = 0; c < kCh; ++c) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (u < dpt) {
                            s0 += qreg[u] * sK[(c0 + c) * D + sub * dpt + u];
                            s1 += doreg[u] * sV[(c0 + c) * D + sub * dpt + u];
                        }
                    ps[c] = s0;
                    pp[c] = s1;
                }
                // dS of the chunk's kept pairs (0 elsewhere), in ps
#pragma unroll
                for (int c = 0; c < kCh; ++c) {
                    const float s = g.scale * group_sum(ps[c]);
                    const float dp = group_sum(pp[c]);
                    const bool keep = valid && c0 + c < rows_b && (!diag || c0 + c <= row + sp.diag_off);
                    const float P = keep ? expf(s - lse_i) : 0.f;
                    ps[c] = P * (dp - delta_i);
                }
#pragma unroll
                for (int c = 0; c < kCh; ++c)
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (u < dpt) acc[u] += ps[c] * sK[(c0 + c) * D + sub * dpt + u];
            }
            if (diag) ++n_part;
            else ++n_full;
        }
        if (!have_next || nxt.r != cur.r) {
            if (tile_stats && threadIdx.x == 0) {
                atomicAdd((unsigned long long *)&tile_stats[cur.r * g.N + d], (unsigned long long)n_full);
                atomicAdd((unsigned long long *)&tile_stats[g.N * g.N + cur.r * g.N + d], (unsigned long long)n_part);
            }
            n_full = n_part = 0;
        }
        cur = nxt;
        have = have_next;
    }
    if (!valid) return;
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (u < dpt) dq[qoff + u] = g.scale * acc[u];
}

// dK, dV: key tile b of stripe e of key/value head blockIdx.y; visits every
// query tile that sees it, for each of the G query heads that read the head,
// in ring order (round r: the key stripe sits on device d = e + r).
template <int DPT>
__global__ void __launch_bounds__(kThreads) simt_dkdv_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ lse, const float *__restrict__ dO, const float *__restrict__ delta,
    float *__restrict__ dk, float *__restrict__ dv, AttnGeom g) {
    extern __shared__ __align__(16) float smem[];
    float *sQ = smem, *sdO = smem + T * g.D;
    float *sL = smem + 2 * T * g.D, *sDel = sL + T;
    constexpr int kU = Dim<DPT>::kU, kCh = grad_chunk<DPT>();
    const Dim<DPT> dm(g.D);
    const int64_t L = g.L;
    const int D = dm.D, dpt = dm.dpt;
    const int nq = (int)((L + T - 1) / T);
    const int bg = nq - 1 - (int)(blockIdx.x % nq);
    const int e = (int)(blockIdx.x / nq);
    const int64_t bh = blockIdx.y;
    const int row = threadIdx.x / kTPR, sub = threadIdx.x % kTPR;  // key row in the tile
    const int64_t j = (int64_t)bg * T + row;
    const SeqSpan sq = seq_of(g.seqs, bg, T, nq);  // packed sequences: own sequence's tiles
    const int b = bg - sq.start, nqs = sq.count;
    const bool valid = j < L;
    const int64_t koff = bh * g.stride_bh + (int64_t)e * g.stripe_stride + j * D + sub * dpt;
    float kreg[kU], vreg[kU], ak[kU], av[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        kreg[u] = (u < dpt && valid) ? k[koff + u] : 0.f;
        vreg[u] = (u < dpt && valid) ? v[koff + u] : 0.f;
        ak[u] = av[u] = 0.f;
    }
    const int rows_b = rows_in_tile(L, bg);
    // the (query head and round, query tile) sequence; the next tile's Q,
    // dO and row statistics load during this one
    struct Cur {
        int hr, a;
        QuerySpan sp;
        const float *q, *dO, *lse, *del;
    };
    auto seek = [&](Cur &c) -> bool {
        for (; c.hr < g.G * g.N; ++c.hr, c.a = -1) {
            const int64_t bq = bh * g.G + c.hr / g.N;  // query head
            const int d = (e + c.hr % g.N) % g.N;       // round r: the key stripe sits on device e + r
            c.sp = query_span(g.layout, d, e, b, nqs, rows_b);
            if (c.a < c.sp.a_lo) c.a = c.sp.a_lo;
            if (c.a < nqs) {
                c.q = q + bq * g.stride_bh + (int64_t)d * g.stripe_stride;
                c.dO = dO + bq * g.stride_bh + (int64_t)d * g.stripe_stride;
                c.lse = lse + bq * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride;
                c.del = delta + bq * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride;
                return true;
            }
        }
        return false;
    };
    auto load_stats = [&](const Cur &c, float &lv, float &dv_) {
        const int ag = sq.start + c.a;
        const bool in = threadIdx.x < rows_in_tile(L, ag);
        lv = (threadIdx.x < T && in) ? c.lse[(int64_t)ag * T + threadIdx.x] : 0.f;
        dv_ = (threadIdx.x < T && in) ? c.del[(int64_t)ag * T + threadIdx.x] : 0.f;
    };
    Cur cur{0, -1, QuerySpan{0, 0, 0}, nullptr, nullptr, nullptr, nullptr};
    bool have = seek(cur);
    TileRegs<DPT> rq, ro;
    float lv = 0.f, dlv = 0.f;
    if (have) {
        tile_load(rq, cur.q, L, dm, sq.start + cur.a);
        tile_load(ro, cur.dO, L, dm, sq.start + cur.a);
        load_stats(cur, lv, dlv);
    }
    while (have) {
        __syncthreads();
        tile_store(rq, sQ, dm);
        tile_store(ro, sdO, dm);
        if (threadIdx.x < T) {
            sL[threadIdx.x] = lv;
            sDel[threadIdx.x] = dlv;
        }
        __syncthreads();
        Cur nxt = cur;
        ++nxt.a;
        const bool have_next = seek(nxt);
        if (have_next) {
            tile_load(rq, nxt.q, L, dm, sq.start + nxt.a);
            tile_load(ro, nxt.dO, L, dm, sq.start + nxt.a);
            load_stats(nxt, lv, dlv);
        }
        {
            const QuerySpan &sp = cur.sp;
            const int rows_a = rows_in_tile(L, sq.start + cur.a);
            const bool diag = sp.has_diag && cur.a == sp.a_lo;
#pragma unroll 1
            for (int c0 = 0; c0 < T; c0 += kCh) {  // query rows c0 + c of the tile
                float ps[kCh], pp[kCh];
#pragma unroll
                for (int c = 0; c < kCh; ++c) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (u < dpt) {
                            s0 += kreg[u] * sQ[(c0 + c) * D + sub * dpt + u];
                            s1 += vreg[u] * sdO[(c0 + c) * D + sub * dpt + u];
                        }
                    ps[c] = s0;
                    pp[c] = s1;
                }
                // P (in pp) and dS (in ps) of the kept pairs, 0 elsewhere: pair
                // (query row c0 + c, key row `row`) kept iff row <= c0 + c + diag_off
#pragma unroll
                for (int c = 0; c < kCh; ++c) {
                    const float s = g.scale * group_sum(ps[c]);
                    const float dp = group_sum(pp[c]);
                    const bool keep = valid && c0 + c < rows_a && (!diag || row <= c0 + c + sp.diag_off);
                    const float P = keep ? expf(s - sL[c0 + c]) : 0.f;
                    ps[c] = P * (dp - sDel[c0 + c]);
                    pp[c] = P;
                }
#pragma unroll
                for (int c = 0; c < kCh; ++c)
#pragma unroll
                    for (int u = 0; u < kU; ++u)
                        if (u < dpt) {
                            ak[u] += ps[c] * sQ[(c0 + c) * D + sub * dpt + u];
                            av[u] += pp[c] * sdO[(c0 + c) * D + sub * dpt + u];
                        }
            }
        }
        cur = nxt;
        have = have_next;
    }
    if (!valid) return;
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (u < dpt) {
            dk[koff + u] = g.scale * ak[u];
            dv[koff + u] = av[u];
        }
}

}  // namespace

int launch_simt_fwd(const float *q, const float *k, const float *v, float *o, float *lse,
                    const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream) {
    const int nq = (int)((g.L + T - 1) / T);
    dim3 grid((unsigned)(nq * g.N), (unsigned)g.BH);
    const size_t smem = 2 * T * g.D * sizeof(float);
    if (g.D == 64)
        simt_fwd_kernel<8><<<grid, kThreads, smem, stream>>>(q, k, v, o, lse, g, tile_stats);
    else if (g.D == 128)
        simt_fwd_kernel<16><<<grid, kThreads, smem, stream>>>(q, k, v, o, lse, g, tile_stats);
    else
        simt_fwd_kernel<0><<<grid, kThreads, smem, stream>>>(q, k, v, o, lse, g, tile_stats);
    return cuda_status(cudaGetLastError());
}

int launch_simt_round(const float *q_d, const float *k_e, const float *v_e, float *o_acc,
                      float *lse_acc, float *o_out, int d, int e, int first, const AttnGeom &g,
                      int64_t *tile_stats, cudaStream_t stream) {
    const int nq = (int)((g.L + T - 1) / T);
    dim3 grid((unsigned)nq, (unsigned)g.BH);
    const size_t smem = 2 * T * g.D * sizeof(float);
    AttnGeom gs = g;
    gs.stripe_stride = 0;
    gs.lse_stripe_stride = 0;
    if (g.D == 64)
        simt_round_kernel<8><<<grid, kThreads, smem, stream>>>(q_d, k_e, v_e, o_acc, lse_acc, o_out, d, e,
                                                              first, gs, tile_stats);
    else if (g.D == 128)
        simt_round_kernel<16><<<grid, kThreads, smem, stream>>>(q_d, k_e, v_e, o_acc, lse_acc, o_out, d, e,
                                                               first, gs, tile_stats);
    else
        simt_round_kernel<0><<<grid, kThreads, smem, stream>>>(q_d, k_e, v_e, o_acc, lse_acc, o_out, d, e,
                                                              first, gs, tile_stats);
    return cuda_status(cudaGetLastError());
}

template <int DPT>
static int launch_simt_grads(const float *q, const float *k, const float *v, const float *lse, const float *dO,
                             float *dq, float *dk, float *dv, const float *delta_ws, const AttnGeom &g,
                             int64_t *tile_stats, cudaStream_t stream) {
    const int nq = (int)((g.L + T - 1) / T);
    dim3 grid((unsigned)(nq * g.N), (unsigned)g.BH);
    const size_t smem = 2 * T * g.D * sizeof(float);
    simt_dq_kernel<DPT><<<grid, kThreads, smem, stream>>>(q, k, v, lse, dO, delta_ws, dq, g, tile_stats);
    const int st = cuda_status(cudaGetLastError());
    if (st != STRIPED_OK) return st;
    dim3 grid_kv((unsigned)(nq * g.N), (unsigned)(g.BH / g.G));  // key tiles of every key/value head
    simt_dkdv_kernel<DPT><<<grid_kv, kThreads, smem + 2 * T * sizeof(float), stream>>>(q, k, v, lse, dO,
                                                                                       delta_ws, dk, dv, g);
    return cuda_status(cudaGetLastError());
}

int launch_simt_bwd(const float *q, const float *k, const float *v, const float *o,
                    const float *lse, const float *dO, float *dq, float *dk, float *dv,
                    float *delta_ws, const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream) {
    // full [BH][S][D] tensors: rows of all heads are contiguous
    const int64_t rows = g.BH * g.N * g.L;
    simt_delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(o, dO, delta_ws, rows, g.D);
    const int st = cuda_status(cudaGetLastError());
    if (st != STRIPED_OK) return st;
    if (g.D == 64) return launch_simt_grads<8>(q, k, v, lse, dO, dq, dk, dv, delta_ws, g, tile_stats, stream);
    if (g.D == 128) return launch_simt_grads<16>(q, k, v, lse, dO, dq, dk, dv, delta_ws, g, tile_stats, stream);
    return launch_simt_grads<0>(q, k, v, lse, dO, dq, dk, dv, delta_ws, g, tile_stats, stream);
}

}  // namespace striped
