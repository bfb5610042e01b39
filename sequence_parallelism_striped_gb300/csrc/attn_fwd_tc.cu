// attn_fwd_tc.cu -- bf16 striped causal attention forward on tcgen05.
//
// Method (pages on "Striped Attention: Faster Ring Attention for Causal
// Transformers"): the query tile of virtual device d visits, in ring rounds
// r = 0..N-1, the key/value stripe e = (d - r) mod N (research.elamur.ai
// summary page, §Summary); under the striped placement about half of every
// round's tiles are masked and skipped (§Summary, second paragraph), and the
// per-round partial results are merged exactly (pith.science paper page,
// abstract) -- here by an online softmax with a log-sum-exp accumulator.
//
// One CTA = one 128-row query tile of one (b, h, stripe); K/V come from the
// key/value head of h (grouped-query attention) and, with packed sequences,
// only from the tiles of the query tile's own sequence.  HD = 128 or 64.
//   warp 0      TMA producer: K/V tiles into a ring of stages (3 at HD = 128)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  softmax + epilogue; thread t owns query row t (TMEM lane t)
//               and first stores that row of Q into TMEM
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O [256,256+HD),
// Q [256+HD,256+3HD/2) as bf16 pairs.
//   S_j = Q K_j^T            (TS MMA: A = Q from TMEM, B = K K-major;
//                             M=N=128, K=16 x 8), so the tensor core reads
//                             only K from shared memory for it
//   P_j = exp2(S_j*c - m) written back over S_j as bf16 (64 columns)
//   O  += P_j V_j            (TS MMA: A = P from TMEM, B = V MN-major)
// S is double-buffered so S_{j+1} runs on the tensor core while the softmax
// warps work on S_j.  The running max is rescaled lazily: O is corrected in
// TMEM only when a row max grows by more than 2^8 (exact, because the final
// normalisation divides by the sum taken against the same reference).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace striped {

namespace {

constexpr int BM = 128, BN = 128;
constexpr uint32_t kBoxBytes = 128 * 128;   // 128 rows x 64 bf16 (one 128-byte-swizzle box)
constexpr int kThreads = 192;

// Shared-memory plan for head dimension HD (64 or 128): K/V tiles of HD/64
// boxes each, in a ring of NS stages (3 at HD = 128, 5 at HD = 64).
template <int HD>
struct FwdCfg {
    static constexpr int kBoxes = HD / 64;
    static constexpr int NS = HD == 128 ? 3 : 5;
    static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
    static constexpr uint32_t kStageBytes = 2 * kTileBytes;  // K + V
    static constexpr uint32_t kBarOff = NS * kStageBytes;
    static constexpr size_t kSmemBytes = 1024 + kBarOff + 256;
    static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
    AttnGeom g;
    const __nv_bfloat16 *q;       // queries (batched: full tensor; round mode: the stripe slice)
    int d_fixed, e_fixed, first;  // single-round mode only
    __nv_bfloat16 *o;             // batched: output
    float *lse;                   // batched: output
    float *o_acc, *lse_acc;       // round mode: accumulator
    __nv_bfloat16 *o_out;         // round mode: optional copy
    int64_t *tile_stats;
    WaitCtl wc;  // status word, wait bound, test hook
};

template <int NS>
struct Bars {
    uint64_t q_full;
    uint64_t kv_full[NS];
    uint64_t kv_empty[NS];
    uint64_t s_full[2];
    uint64_t p_ready;
    uint64_t o_done;
    uint64_t drain;  // every MMA of the issuer has completed (before TMEM is freed)
    uint32_t tmem_slot;
};

__device__ __forceinline__ int tile_rows(int64_t L, int t) {
    const int64_t r = L - (int64_t)t * BM;
    return r >= BM ? BM : (int)r;
}

// kPacked: packed variable-length sequences (the sequence table is
// consulted); the dense instantiation compiles the span as {0, nq}.
template <int HD, bool kRound, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const FwdParams p) {
    using Cfg = FwdCfg<HD>;
    constexpr int NS = Cfg::NS;
    constexpr uint32_t kTileBytes = Cfg::kTileBytes, kStageBytes = Cfg::kStageBytes, kKVOff = 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    Bars<NS> *bars = reinterpret_cast<Bars<NS> *>(smem + Cfg::kBarOff);
    const uint32_t sbase = smem_u32(smem);
    const AttnGeom &g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int nq = (int)((g.L + BM - 1) / BM);
    int ag, d;  // ag: tile index in the device's slice
    int64_t bh;
    if (kRound) {
        ag = nq - 1 - (int)blockIdx.x;
        d = p.d_fixed;
        bh = blockIdx.y;
    } else {
        // Head-major order: the CTAs resident at one time belong to one head
        // and share its K/V tiles in L2.  Within a head the heaviest query
        // tiles go first (largest a; for contiguous also largest d).
        const int64_t id = blockIdx.x;
        const int64_t per_head = (int64_t)nq * g.N;
        bh = id / per_head;
        const int rem = (int)(id % per_head);
        ag = nq - 1 - rem / g.N;
        const int dd = rem % g.N;
        d = (g.layout == STRIPED_LAYOUT_CONTIGUOUS) ? g.N - 1 - dd : dd;
    }
    const int rows_a = tile_rows(g.L, ag);
    // packed sequences: the schedule works on tiles of the query tile's own
    // sequence (tiles sq.start .. sq.start + nqs - 1 of every slice)
    const SeqSpan sq = kPacked ? seq_of(g.seqs, ag, BM, nq) : SeqSpan{0, nq};
    const int a = ag - sq.start;  // tile index inside the sequence
    const int nqs = sq.count;
    const int nrounds = kRound ? 1 : g.N;
    const int e_fixed = p.e_fixed;
    // Key stripes are visited in the same global order e = 0..N-1 by every
    // query tile (so resident CTAs read the same key tiles at the same
    // time); tile counts are still attributed to ring round (d - e) mod N.
    // The first tile (e = 0, b = 0) always holds a kept key for every row.
    auto stripe_of = [=](int r) { return kRound ? e_fixed : r; };

    // number of key tiles this query tile visits
    int nt = 0;
    for (int r = 0; r < nrounds; ++r) {
        const RoundSpan sp = round_span(g.layout, d, stripe_of(r), a, nqs, rows_a);
        nt += sp.nfull + sp.has_diag;
    }

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 4);  // the four softmax warps stored Q in TMEM
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->s_full[0]), 1);
        mbar_init(smem_u32(&bars->s_full[1]), 1);
        mbar_init(smem_u32(&bars->p_ready), 4);
        mbar_init(smem_u32(&bars->o_done), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    const uint32_t tS0 = tmem, tS1 = tmem + 128, tO = tmem + 256, tQ = tmem + 256 + HD;

    const int qstripe = kRound ? 0 : d;
    const int kvh = (int)(bh / g.G);  // key/value head read by query head bh
    if (warp == 0 && lane == 0 && nt > 0) {
        // ---------------- TMA producer
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        // test hook: the first K/V tile is never loaded, so every wait on it
        // runs out (the kernel must then record the timeout and return)
        const bool skip_first = p.wc.inject == kInjectFwdSkipKV;
        int j = 0;
        bool ok = true;
        for (int r = 0; r < nrounds && ok; ++r) {
            const int e = stripe_of(r);
            const int kstripe = kRound ? 0 : e;
            const RoundSpan sp = round_span(g.layout, d, e, a, nqs, rows_a);
            const int ntr = sp.nfull + sp.has_diag;
            for (int b = 0; b < ntr; ++b, ++j) {
                const int s = j % NS;
                const int kb = sq.start + b;  // key tile in the slice
                if (j >= NS && !mbar_wait(smem_u32(&bars->kv_empty[s]), ((j / NS) + 1) & 1, p.wc)) {
                    ok = false;
                    break;
                }
                if (skip_first && j == 0) continue;
                const uint32_t fb = smem_u32(&bars->kv_full[s]);
                const uint32_t kdst = sbase + kKVOff + s * kStageBytes;
                const uint32_t vdst = kdst + kTileBytes;
                mbar_arrive_expect_tx(fb, 2 * kTileBytes);
#pragma unroll
                for (int x = 0; x < Cfg::kBoxes; ++x) {
                    tma_load_4d(kdst + x * kBoxBytes, &tmK, fb, 64 * x, kb * BN, kstripe, kvh);
                    tma_load_4d(vdst + x * kBoxBytes, &tmV, fb, 64 * x, kb * BN, kstripe, kvh);
                }
            }
        }
        // loads [0, j) were issued: wait (bounded) for the last of each stage,
        // so that on an error path none lands after the CTA has exited
        for (int t = j > NS ? j - NS : 0; t < j; ++t)
            if (!(skip_first && t == 0)) mbar_wait(smem_u32(&bars->kv_full[t % NS]), (t / NS) & 1, p.wc);
    } else if (warp == 1 && lane == 0 && nt > 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, HD, false, true);
        bool ok = mbar_wait(smem_u32(&bars->q_full), 0, p.wc);
        tc_fence_after();
        auto issue_s = [&](int t) -> bool {
            const int s = t % NS;
            if (!mbar_wait(smem_u32(&bars->kv_full[s]), (t / NS) & 1, p.wc)) return false;
            tc_fence_after();
            const uint32_t kaddr = sbase + kKVOff + s * kStageBytes;
            const uint32_t dS = (t & 1) ? tS1 : tS0;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                mma_ts(dS, tQ + kk * 8, sdesc_sw128(kaddr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->s_full[t & 1]));
            return true;
        };
        if (ok) ok = issue_s(0);
        if (ok && nt > 1) ok = issue_s(1);
        for (int j = 0; j < nt && ok; ++j) {
            if (!mbar_wait(smem_u32(&bars->p_ready), j & 1, p.wc)) break;
            tc_fence_after();
            const int s = j % NS;
            const uint32_t vaddr = sbase + kKVOff + s * kStageBytes + kTileBytes;
            const uint32_t tP = (j & 1) ? tS1 : tS0;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(tO, tP + kk * 8, sdesc_sw128(vaddr + kk * 2048, kBoxBytes, 1024), idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
            // only stages the producer will refill get a release (no arrival
            // may land after the CTA has exited)
            if (j + NS < nt) mma_commit(smem_u32(&bars->kv_empty[s]));
            mma_commit(smem_u32(&bars->o_done));
            if (j + 2 < nt) ok = issue_s(j + 2);
        }
        // every MMA issued above completes before TMEM is freed (error paths)
        mma_commit(smem_u32(&bars->drain));
        mbar_wait(smem_u32(&bars->drain), 0, p.wc);
    } else if (warp >= 2) {
        // ---------------- softmax + epilogue
        const int quarter = warp & 3;
        const int ri = quarter * 32 + lane;  // query row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float cl2 = g.scale * 1.4426950408889634f;  // scores -> log2 units
        if (nt > 0) {
            // Q row ri -> TMEM columns [tQ, tQ + 64) as bf16 pairs: the A
            // operand of every S = Q K^T, so the tensor core reads only K
            // from shared memory for it
            const int64_t qrow = (int64_t)ag * BM + ri;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.q + bh * g.stride_bh + (int64_t)qstripe * g.stripe_stride + qrow * HD);
#pragma unroll
            for (int h = 0; h < HD / 64; ++h) {  // 64 bf16 = 32 columns per chunk
                uint32_t qa[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 w = qrow < g.L ? __ldg(src + 8 * h + v) : make_uint4(0u, 0u, 0u, 0u);
                    qa[4 * v] = w.x, qa[4 * v + 1] = w.y, qa[4 * v + 2] = w.z, qa[4 * v + 3] = w.w;
                }
                tmem_st32(tQ + lane_off + 32 * h, qa);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->q_full));
        }
        float m_ref = -INFINITY, l = 0.f;
        int j = 0;
        bool ok = true;
        for (int r = 0; r < nrounds && ok; ++r) {
            const int e = stripe_of(r);
            const RoundSpan sp = round_span(g.layout, d, e, a, nqs, rows_a);
            const int ntr = sp.nfull + sp.has_diag;
            int n_full = 0, n_part = 0;  // tiles of this round turned into P below
            for (int b = 0; b < ntr; ++b, ++j) {
                const uint32_t tS = ((j & 1) ? tS1 : tS0) + lane_off;
                if (!mbar_wait(smem_u32(&bars->s_full[j & 1]), (j >> 1) & 1, p.wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float sv[BN];
                {
                    // all four loads in flight before one wait
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    tmem_ld32(tS, r0);
                    tmem_ld32(tS + 32, r1);
                    tmem_ld32(tS + 64, r2);
                    tmem_ld32(tS + 96, r3);
                    tmem_ld_wait(r0);
                    tmem_ld_wait(r1);
                    tmem_ld_wait(r2);
                    tmem_ld_wait(r3);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        sv[u] = __uint_as_float(r0[u]);
                        sv[32 + u] = __uint_as_float(r1[u]);
                        sv[64 + u] = __uint_as_float(r2[u]);
                        sv[96 + u] = __uint_as_float(r3[u]);
                    }
                }
                const bool diag = sp.has_diag && b == sp.nfull;
                const int kv_valid = tile_rows(g.L, sq.start + b);
                if (diag || kv_valid < BN) {
                    const int lim = diag ? min(ri + sp.diag_off, kv_valid - 1) : kv_valid - 1;
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c > lim) sv[c] = -INFINITY;
                }
                // row max as 8 independent chains of three-input max (a
                // single chain of 128 dependent max operations would be pure
                // latency)
                float mx8[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx8[t] = sv[t];
#pragma unroll
                for (int c = 8; c < BN; c += 16)
#pragma unroll
                    for (int t = 0; t < 8; ++t) mx8[t] = fmax3(mx8[t], sv[c + t], sv[c + 8 + t]);
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float m_tile = mx * cl2;
                // lazy rescale: move the reference only when the max grows a lot
                bool move = (j == 0) ? true : (m_tile > m_ref + kRescaleThreshold);
                const float m_new = move ? fmaxf(m_ref, m_tile) : m_ref;
                const float alpha = (j == 0 || !move) ? 1.f : ex2(m_ref - m_new);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                // exponent arguments two at a time (paired fp32 FMA), the row
                // sum in four paired accumulators
                const uint64_t cl2x2 = f2(cl2, cl2), nm2 = f2(-m_use, -m_use);
                uint64_t acc4[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pk[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 2; ++c) {
                    const float2 x = f2_split(fma2(f2(sv[2 * c], sv[2 * c + 1]), cl2x2, nm2));
                    const float p0 = ex2(x.x), p1 = ex2(x.y);
                    acc4[c & 3] = add2(acc4[c & 3], f2(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                const float2 s01 = f2_split(add2(acc4[0], acc4[1])), s23 = f2_split(add2(acc4[2], acc4[3]));
                const float sum = (s01.x + s01.y) + (s23.x + s23.y);
                {
                    uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
                    uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
                    tmem_st32(tS, lo);
                    tmem_st32(tS + 32, hi);
                }
                tmem_st_wait();
                l = l * alpha + sum;
                m_ref = m_new;
                if (j > 0) {
                    // PV_{j-1} must be complete before O is touched or PV_j issued
                    if (!mbar_wait(smem_u32(&bars->o_done), (j - 1) & 1, p.wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t rr[32];
                            tmem_ld32(tO + lane_off + c * 32, rr);
                            tmem_ld_wait(rr);
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                rr[u] = __float_as_uint(__uint_as_float(rr[u]) * alpha);
                            tmem_st32(tO + lane_off + c * 32, rr);
                        }
                        tmem_st_wait();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready));
                if (diag) ++n_part;
                else ++n_full;
            }
            // the round's counters get the tiles that ran (one thread)
            if (p.tile_stats && warp == 2 && lane == 0 && (n_full | n_part)) {
                const int rr = ring_round_of(d, e, g.N);
                atomicAdd((unsigned long long *)&p.tile_stats[rr * g.N + d], (unsigned long long)n_full);
                atomicAdd((unsigned long long *)&p.tile_stats[g.N * g.N + rr * g.N + d], (unsigned long long)n_part);
            }
        }
        // ---------------- epilogue
        if (ok && nt > 0) {
            ok = mbar_wait(smem_u32(&bars->o_done), (nt - 1) & 1, p.wc);
            tc_fence_after();
        }
        const int64_t i = (int64_t)ag * BM + ri;
        const bool valid_row = i < g.L;
        const bool empty = !(l > 0.f) || !ok;
        const float inv_l = empty ? 0.f : 1.f / l;
        const float lse_row = empty ? -INFINITY : (m_ref + log2f(l)) * 0.6931471805599453f;
        const int64_t orow = (int64_t)bh * g.stride_bh + (int64_t)d * g.stripe_stride + i * HD;
        if (!kRound) {
            if (valid_row) p.lse[bh * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride + i] = lse_row;
        }
        float lse_a = -INFINITY, wa = 0.f, wr = 1.f, lse_new = lse_row;
        if (kRound && valid_row) {
            float *lp = p.lse_acc + bh * g.lse_stride_bh + i;
            lse_a = p.first ? -INFINITY : *lp;
            const float mxl = fmaxf(lse_a, lse_row);
            if (mxl == -INFINITY) {
                wa = p.first ? 0.f : 1.f;
                wr = 0.f;
                lse_new = -INFINITY;
            } else {
                wa = expf(lse_a - mxl);
                wr = expf(lse_row - mxl);
                lse_new = mxl + logf(wa + wr);
                const float inv = 1.f / (wa + wr);
                wa *= inv;
                wr *= inv;
            }
        }
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
            uint32_t rr[32];
            if (nt > 0) {
                tmem_ld32(tO + lane_off + c * 32, rr);
                tmem_ld_wait(rr);
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) rr[u] = 0u;
            }
            if (!valid_row) continue;
            if (!kRound) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow + c * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * inv_l, __uint_as_float(rr[8 * v + 1]) * inv_l);
                    w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * inv_l, __uint_as_float(rr[8 * v + 3]) * inv_l);
                    w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * inv_l, __uint_as_float(rr[8 * v + 5]) * inv_l);
                    w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * inv_l, __uint_as_float(rr[8 * v + 7]) * inv_l);
                    dst[v] = w;
                }
            } else {
                const int64_t arow = (int64_t)bh * g.stride_bh + i * HD + c * 32;
                float4 *acc = reinterpret_cast<float4 *>(p.o_acc + arow);
                float vals[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    float4 prev = p.first ? make_float4(0.f, 0.f, 0.f, 0.f) : acc[v];
                    vals[4 * v + 0] = wa * prev.x + wr * __uint_as_float(rr[4 * v + 0]) * inv_l;
                    vals[4 * v + 1] = wa * prev.y + wr * __uint_as_float(rr[4 * v + 1]) * inv_l;
                    vals[4 * v + 2] = wa * prev.z + wr * __uint_as_float(rr[4 * v + 2]) * inv_l;
                    vals[4 * v + 3] = wa * prev.w + wr * __uint_as_float(rr[4 * v + 3]) * inv_l;
                    acc[v] = make_float4(vals[4 * v], vals[4 * v + 1], vals[4 * v + 2], vals[4 * v + 3]);
                }
                if (p.o_out) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o_out + arow);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(vals[8 * v + 0], vals[8 * v + 1]);
                        w.y = pack_bf16x2(vals[8 * v + 2], vals[8 * v + 3]);
                        w.z = pack_bf16x2(vals[8 * v + 4], vals[8 * v + 5]);
                        w.w = pack_bf16x2(vals[8 * v + 6], vals[8 * v + 7]);
                        dst[v] = w;
                    }
                }
            }
        }
        if (kRound && valid_row) p.lse_acc[bh * g.lse_stride_bh + i] = lse_new;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

template <int HD>
static int set_smem_once() {
    static PerDeviceOnce once;
    return once.get([] {
        const int bytes = (int)FwdCfg<HD>::kSmemBytes;
        const cudaError_t e[3] = {
            cudaFuncSetAttribute(tc_fwd_kernel<HD, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
            cudaFuncSetAttribute(tc_fwd_kernel<HD, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
            cudaFuncSetAttribute(tc_fwd_kernel<HD, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)};
        int status = STRIPED_OK;
        for (cudaError_t x : e)
            if (x != cudaSuccess) status = cuda_status(x);
        return status;
    });
}

template <int HD>
static int launch_fwd_hd(const CUtensorMap &mk, const CUtensorMap &mv, const FwdParams &p, int64_t nblocks,
                         cudaStream_t stream) {
    const int st = set_smem_once<HD>();
    if (st != STRIPED_OK) return st;
    const size_t bytes = FwdCfg<HD>::kSmemBytes;
    if (p.g.seqs.n > 0)
        tc_fwd_kernel<HD, false, true><<<(unsigned)nblocks, kThreads, bytes, stream>>>(mk, mv, p);
    else
        tc_fwd_kernel<HD, false, false><<<(unsigned)nblocks, kThreads, bytes, stream>>>(mk, mv, p);
    return cuda_status(cudaGetLastError());
}

template <int HD>
static int launch_round_hd(const CUtensorMap &mk, const CUtensorMap &mv, const FwdParams &p, dim3 grid,
                           cudaStream_t stream) {
    const int st = set_smem_once<HD>();
    if (st != STRIPED_OK) return st;
    tc_fwd_kernel<HD, true, false><<<grid, kThreads, FwdCfg<HD>::kSmemBytes, stream>>>(mk, mv, p);
    return cuda_status(cudaGetLastError());
}

int launch_tc_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                  const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream) {
    if (fwd_pair_eligible(g, device_sm_count())) return launch_tc_fwd_pair(q, k, v, o, lse, g, tile_stats, stream);
    int st = STRIPED_OK;
    CUtensorMap mk, mv;
    const int64_t bh_kv = g.BH / g.G;
    if ((st = make_bf16_map(&mk, k, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mv, v, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)))
        return st;
    FwdParams p{};
    p.g = g;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.o = reinterpret_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nq = (g.L + BM - 1) / BM;
    const int64_t nblocks = nq * g.N * g.BH;
    if (nblocks > 0x7fffffffll) return STRIPED_ERR_UNSUPPORTED;
    return g.D == 64 ? launch_fwd_hd<64>(mk, mv, p, nblocks, stream) : launch_fwd_hd<128>(mk, mv, p, nblocks, stream);
}

int launch_tc_round(const void *q_d, const void *k_e, const void *v_e, float *o_acc, float *lse_acc,
                    void *o_out, int d, int e, int first, const AttnGeom &g, int64_t *tile_stats,
                    cudaStream_t stream) {
    int st = STRIPED_OK;
    CUtensorMap mk, mv;
    // the slices are single stripes: a stripe dimension of extent 1
    if ((st = make_bf16_map(&mk, k_e, g.D, g.L, 1, g.BH, g.L * g.D, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mv, v_e, g.D, g.L, 1, g.BH, g.L * g.D, g.stride_bh, 128)))
        return st;
    FwdParams p{};
    p.g = g;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q_d);
    p.g.G = 1;
    p.g.stripe_stride = 0;
    p.g.lse_stripe_stride = 0;
    p.d_fixed = d;
    p.e_fixed = e;
    p.first = first;
    p.o_acc = o_acc;
    p.lse_acc = lse_acc;
    p.o_out = reinterpret_cast<__nv_bfloat16 *>(o_out);
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nq = (g.L + BM - 1) / BM;
    if (g.BH > 65535) return STRIPED_ERR_UNSUPPORTED;
    dim3 grid((unsigned)nq, (unsigned)g.BH);
    return g.D == 64 ? launch_round_hd<64>(mk, mv, p, grid, stream) : launch_round_hd<128>(mk, mv, p, grid, stream);
}

}  // namespace striped
