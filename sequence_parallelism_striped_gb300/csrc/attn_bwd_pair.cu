// attn_bwd_pair.cu -- bf16 striped causal attention backward on a CTA pair
// (tcgen05 cta_group::2): two key tiles per cluster of two CTAs.
//
// Same mathematics as attn_bwd_tc.cu (the derivative of the exact causal
// attention of the forward; P = exp(scale q k^T - LSE), Delta = <dO, O>):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),
//   dK = scale * dS^T Q,  dQ = scale * dS K,
// with the ring schedule of the striped placement (research.elamur.ai
// summary page, §Summary): key tile b of stripe e is seen by query tiles
// a >= b of every query stripe d, the diagonal tile a = b keeping
// j <= i + [e <= d] - 1.  Key tile b of stripes e and e+1 are seen by the
// same query tiles (only the diagonal mask differs), so one cluster of two
// CTAs takes both: CTA r holds key tile b of stripe e0 + r and its dK, dV,
// and the pair sweeps the query tiles together.
//
// Why a pair.  A one-CTA backward sends, per 128 x 128 tile pair, a 64 KB
// fp32 partial of dQ_i = dS_i K to the global accumulator; that L2
// reduction traffic limits it.  Here dQ_i is contracted over the pair's 256
// keys on the tensor core (an M = 128 paired MMA: CTA r computes query rows
// [64r, 64r+64) of the tile from the dS of BOTH key tiles), so each key tile
// reduces 32 KB instead of 64 KB.  The other four products are M = 256
// paired MMAs (each CTA supplies its 128 key rows of A and half of B), which
// also halves what each CTA reads of Q_i and dO_i as B operands.
//
// Shared memory of CTA r (same offsets in both; the paired MMA reads its
// operands at the same offsets in both CTAs):
//   K, V        own key tile, K-major A of S^T = K Q^T and dP^T = V dO^T
//   KQ          head-dimension half r of K for both key tiles (B of dQ)
//   dS          own dS^T [128 keys][128 queries] (K-major A of dK)
//   dSX         query half r of dS for both key tiles (MN-major A of dQ);
//               each CTA writes the other's half through distributed shared
//               memory
//   QS, dOP     query rows [64r, 64r+64) of Q_i / dO_i (B of S^T / dP^T)
//   QK, dOV     head-dimension half r of Q_i / dO_i (B of dK / dV)
//   statistics  two stages of [LSE*log2e 128 | Delta 128]
// One stage per operand stream: each is refilled as soon as its MMA
// completes, a whole tile (five MMAs) ahead of its next use.
// Tensor memory (both CTAs, 512 columns): S^T [0,128) (P^T bf16 pairs over
// it), dP^T [128,256) (dQ_i over its first 64 columns: lane l holds query
// row l % 64 of the CTA's half, head-dimension columns 64*(l/64) .. +63),
// dV [256,384), dK [384,512).
// Warps: 0 (first CTA) TMA of K, V, KQ and the QS stream for both CTAs;
// 1 tensor-memory allocation (both CTAs) and, in the first CTA, the MMA
// issuer; 2 (first CTA) TMA of the QK, dOP and dOV streams; 3 the
// statistics of its own CTA; 4..11 compute (thread t of warpgroup w owns key
// row t, query columns [64w, 64w+64)).
// MMA order per query tile i: dV_i, S_{i+1}, dQ_i, dK_i, dP_{i+1}.  dQ_i
// leaves through TMA bulk reduce-adds staged in the own dS tile once dK_i
// has read it (per warp, the 4 KB the warp itself writes).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace striped {

namespace {

constexpr int PT = 128;                         // tile edge (keys, queries), head dimension
constexpr uint32_t kBox = 128 * 128;            // 128 rows x 64 bf16 (one 128-byte-swizzle box)
constexpr uint32_t kHalfBox = 64 * 128;         // 64 rows x 64 bf16
constexpr uint32_t kStatBytes = 2 * 128 * 4;
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = 2 * kBox;
constexpr uint32_t kOffKQ = 4 * kBox;           // [key tile of stripe e0 | of e0 + 1]
constexpr uint32_t kOffDS = 6 * kBox;           // [queries 0..63 | 64..127]
constexpr uint32_t kOffDSX = 8 * kBox;          // [key tile of stripe e0 | of e0 + 1]
constexpr uint32_t kOffQS = 10 * kBox;          // [head dims 0..63 | 64..127], 64 rows each
constexpr uint32_t kOffQK = kOffQS + 2 * kHalfBox;
constexpr uint32_t kOffDOP = kOffQK + kBox;
constexpr uint32_t kOffDOV = kOffDOP + 2 * kHalfBox;
constexpr uint32_t kOffStat = kOffDOV + kBox;
constexpr uint32_t kOffBar = kOffStat + 2 * kStatBytes;
constexpr size_t kPairSmemBytes = kOffBar + 256;  // the dynamic smem base is 1024-aligned
static_assert(kPairSmemBytes <= 232448, "shared memory over the per-block limit");
constexpr int kPairThreads = 384;
constexpr uint16_t kBothCtas = 3;

struct PairBars {
    uint64_t kv_full;                                   // first CTA: K, V, KQ of both CTAs landed
    uint64_t qs_full, qs_empty, qk_full, qk_empty;      // first CTA: Q_i streams
    uint64_t dop_full, dop_empty, dov_full, dov_empty;  // first CTA: dO_i streams
    uint64_t p_ready, ds_ready, dq_free;                // first CTA: 16 compute warps of the pair
    uint64_t s_full, dp_full, dq_full, dk_done, acc_done;  // each CTA: paired-MMA completions
    uint64_t st_full[2], st_empty[2];                   // each CTA: its statistics stream
    uint64_t drain;                                     // first CTA: every MMA has completed
    uint32_t tmem_slot;
};
static_assert(sizeof(PairBars) <= 256, "barrier block");

struct PairParams {
    AttnGeom g;
    const float *stats;  // [BH][N][nq][LSE*log2e 128 | Delta 128]
    float *dq_acc;       // [BH][S][D] fp32
    __nv_bfloat16 *dk, *dv;
    int64_t *tile_stats;
    WaitCtl wc;  // status word, wait bound, test hook
};

// Query tiles of key tile b (stripe e) in visiting order: the G query heads
// of the key/value head, per head the stripes d = 0..N-1, per stripe the
// tiles a = nq-1 down to b (tile b holding the diagonal).
struct PairIter {
    int h, d, a;
};

__device__ __forceinline__ void piter_next(PairIter &it, int N, int b, int nq) {
    if (--it.a < b) {
        it.a = nq - 1;
        if (++it.d == N) {
            it.d = 0;
            ++it.h;
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    tc_bwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQh,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO, const __grid_constant__ CUtensorMap tmdOh,
                       const __grid_constant__ CUtensorMap tmdQ, const PairParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if ((smem_u32(smem) & 1023u) != 0) {  // the same in both CTAs: both leave here
        if (threadIdx.x == 0) record_error(p.wc.st, STRIPED_ERR_ALIGN);
        return;
    }
    PairBars *bars = reinterpret_cast<PairBars *>(smem + kOffBar);
    const uint32_t sbase = smem_u32(smem);
    const AttnGeom &g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();  // 0: issues the paired MMAs
    const int N = g.N, G = (int)g.G;
    const int nq = (int)(g.L / PT);

    // Head-major order; within a head the heaviest key tiles (small b) first.
    const int npair = N / 2;
    const int64_t cid = blockIdx.x >> 1;
    const int64_t per_head = (int64_t)nq * npair;
    const int64_t bh = cid / per_head;  // key/value head
    const int rem = (int)(cid % per_head);
    const int b = rem / npair;
    const int e0 = 2 * (rem % npair);
    const int e = e0 + (int)rank;  // this CTA's key stripe
    const int nt = G * N * (nq - b);

    auto bar = [&](const uint64_t &x) { return smem_u32(&x); };
    if (threadIdx.x == 0) {
        mbar_init(bar(bars->kv_full), 1);
        mbar_init(bar(bars->qs_full), 1);
        mbar_init(bar(bars->qs_empty), 1);
        mbar_init(bar(bars->qk_full), 1);
        mbar_init(bar(bars->qk_empty), 1);
        mbar_init(bar(bars->dop_full), 1);
        mbar_init(bar(bars->dop_empty), 1);
        mbar_init(bar(bars->dov_full), 1);
        mbar_init(bar(bars->dov_empty), 1);
        mbar_init(bar(bars->p_ready), 16);
        mbar_init(bar(bars->ds_ready), 16);
        mbar_init(bar(bars->dq_free), 16);
        mbar_init(bar(bars->s_full), 1);
        mbar_init(bar(bars->dp_full), 1);
        mbar_init(bar(bars->dq_full), 1);
        mbar_init(bar(bars->dk_done), 1);
        mbar_init(bar(bars->acc_done), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(bars->st_full[s]), 1);
            mbar_init(bar(bars->st_empty[s]), 8);
        }
        mbar_init(bar(bars->drain), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&bars->tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // barriers of both CTAs initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;

    if (rank == 0 && warp == 0 && lane == 0 && nt > 0) {
        // ---------------- TMA: K, V, KQ once, then the QS stream (both CTAs)
        tma_prefetch_desc(&tmQh);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const uint32_t kvb = bar(bars->kv_full), kvb_cl = mapa_shared(kvb, 0);
        mbar_arrive_expect_tx(kvb, 2 * 6 * kBox);
        for (uint32_t cc = 0; cc < 2; ++cc) {
            const uint32_t dst = mapa_shared(sbase, cc);
            for (int x = 0; x < 2; ++x) {
                tma_load_4d_pair(dst + kOffK + x * kBox, &tmK, kvb_cl, 64 * x, b * PT, e0 + (int)cc, (int)bh);
                tma_load_4d_pair(dst + kOffV + x * kBox, &tmV, kvb_cl, 64 * x, b * PT, e0 + (int)cc, (int)bh);
                tma_load_4d_pair(dst + kOffKQ + x * kBox, &tmK, kvb_cl, 64 * (int)cc, b * PT, e0 + x, (int)bh);
            }
        }
        // test hook: the first QS tile is never loaded, so every wait on it
        // runs out (the kernel must then record the timeout and return)
        const bool skip_first = p.wc.inject == kInjectBwdSkipQ;
        const uint32_t fb = bar(bars->qs_full), fb_cl = mapa_shared(fb, 0);
        PairIter it{0, 0, nq - 1};
        int i = 0;
        for (; i < nt; ++i, piter_next(it, N, b, nq)) {
            if (i > 0 && !mbar_wait_cl(bar(bars->qs_empty), (i - 1) & 1, p.wc)) break;
            if (skip_first && i == 0) continue;
            const int bq = (int)(bh * G + it.h);
            mbar_arrive_expect_tx(fb, 2 * 2 * kHalfBox);
            for (uint32_t cc = 0; cc < 2; ++cc) {
                const uint32_t dst = mapa_shared(sbase, cc);
                for (int x = 0; x < 2; ++x)
                    tma_load_4d_pair(dst + kOffQS + x * kHalfBox, &tmQh, fb_cl, 64 * x, it.a * PT + 64 * (int)cc,
                                     it.d, bq);
            }
        }
        // the last loads issued complete before the pair can exit (bounded)
        mbar_wait_cl(kvb, 0, p.wc);
        if (i > 0 && !(skip_first && i == 1)) mbar_wait_cl(fb, (i - 1) & 1, p.wc);
    } else if (rank == 0 && warp == 2 && lane == 0 && nt > 0) {
        // ---------------- TMA: the dOP, dOV and QK streams (both CTAs), in
        // the order their buffers are released (dP_i, dV_i, dK_i)
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmdOh);
        const uint32_t fop = bar(bars->dop_full), fov = bar(bars->dov_full), fqk = bar(bars->qk_full);
        const uint32_t fop_cl = mapa_shared(fop, 0), fov_cl = mapa_shared(fov, 0), fqk_cl = mapa_shared(fqk, 0);
        PairIter it{0, 0, nq - 1};
        int n_op = 0, n_ov = 0, n_qk = 0;  // tiles issued per stream
        for (int i = 0; i < nt; ++i, piter_next(it, N, b, nq)) {
            const int bq = (int)(bh * G + it.h);
            if (i > 0 && !mbar_wait_cl(bar(bars->dop_empty), (i - 1) & 1, p.wc)) break;
            mbar_arrive_expect_tx(fop, 2 * 2 * kHalfBox);
            for (uint32_t cc = 0; cc < 2; ++cc) {
                const uint32_t dst = mapa_shared(sbase, cc);
                for (int x = 0; x < 2; ++x)
                    tma_load_4d_pair(dst + kOffDOP + x * kHalfBox, &tmdOh, fop_cl, 64 * x, it.a * PT + 64 * (int)cc,
                                     it.d, bq);
            }
            ++n_op;
            if (i > 0 && !mbar_wait_cl(bar(bars->dov_empty), (i - 1) & 1, p.wc)) break;
            mbar_arrive_expect_tx(fov, 2 * kBox);
            for (uint32_t cc = 0; cc < 2; ++cc)
                tma_load_4d_pair(mapa_shared(sbase, cc) + kOffDOV, &tmdO, fov_cl, 64 * (int)cc, it.a * PT, it.d, bq);
            ++n_ov;
            if (i > 0 && !mbar_wait_cl(bar(bars->qk_empty), (i - 1) & 1, p.wc)) break;
            mbar_arrive_expect_tx(fqk, 2 * kBox);
            for (uint32_t cc = 0; cc < 2; ++cc)
                tma_load_4d_pair(mapa_shared(sbase, cc) + kOffQK, &tmQ, fqk_cl, 64 * (int)cc, it.a * PT, it.d, bq);
            ++n_qk;
        }
        if (n_op > 0) mbar_wait_cl(fop, (n_op - 1) & 1, p.wc);
        if (n_ov > 0) mbar_wait_cl(fov, (n_ov - 1) & 1, p.wc);
        if (n_qk > 0) mbar_wait_cl(fqk, (n_qk - 1) & 1, p.wc);
    } else if (warp == 3 && lane == 0 && nt > 0) {
        // ---------------- statistics of each query tile into this CTA (2 stages)
        PairIter it{0, 0, nq - 1};
        int i = 0;
        for (; i < nt; ++i, piter_next(it, N, b, nq)) {
            const int s = i & 1;
            if (i >= 2 && !mbar_wait(bar(bars->st_empty[s]), ((i >> 1) + 1) & 1, p.wc)) break;
            const int64_t bq = bh * G + it.h;
            mbar_arrive_expect_tx(bar(bars->st_full[s]), kStatBytes);
            bulk_load(sbase + kOffStat + s * kStatBytes, p.stats + (((bq * N + it.d) * (int64_t)nq + it.a) << 8),
                      kStatBytes, bar(bars->st_full[s]));
        }
        for (int t = i > 2 ? i - 2 : 0; t < i; ++t) mbar_wait(bar(bars->st_full[t & 1]), (t >> 1) & 1, p.wc);
    } else if (rank == 0 && warp == 1 && lane == 0 && nt > 0) {
        // ---------------- paired-MMA issuer
        constexpr uint32_t id_s = idesc_bf16_f32(2 * PT, PT, false, false);  // S^T, dP^T (M = 256)
        constexpr uint32_t id_kv = idesc_bf16_f32(2 * PT, PT, false, true);  // dV (A in TMEM), dK (M = 256)
        constexpr uint32_t id_q = idesc_bf16_f32(PT, PT, true, true);        // dQ (M = 128)
        auto issue_s = [&](int t) -> bool {
            if (!mbar_wait_cl(bar(bars->qs_full), t & 1, p.wc)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss_pair(tS, sdesc_sw128(sbase + kOffK + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                            sdesc_sw128(sbase + kOffQS + (kk >> 2) * kHalfBox + (kk & 3) * 32, 16, 1024), id_s,
                            kk > 0 ? 1u : 0u);
            mma_commit_pair_mc(bar(bars->s_full), kBothCtas);
            mma_commit_pair(bar(bars->qs_empty));
            return true;
        };
        auto issue_dp = [&](int t) -> bool {
            if (!mbar_wait_cl(bar(bars->dop_full), t & 1, p.wc)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss_pair(tdP, sdesc_sw128(sbase + kOffV + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                            sdesc_sw128(sbase + kOffDOP + (kk >> 2) * kHalfBox + (kk & 3) * 32, 16, 1024), id_s,
                            kk > 0 ? 1u : 0u);
            mma_commit_pair_mc(bar(bars->dp_full), kBothCtas);
            mma_commit_pair(bar(bars->dop_empty));
            return true;
        };
        // tiles whose five MMAs were issued, per query stripe, for both key
        // stripes of the pair: added to the (round, device) counters when the
        // stripe changes (the diagonal tile a = b is the partial one)
        PairIter it{0, 0, nq - 1};
        int cnt_d = -1, n_full = 0, n_part = 0;
        auto flush_counts = [&]() {
            if (p.tile_stats && cnt_d >= 0 && (n_full | n_part)) {
                for (int x = 0; x < 2; ++x) {
                    const int rr = ring_round_of(cnt_d, e0 + x, N);
                    atomicAdd((unsigned long long *)&p.tile_stats[rr * N + cnt_d], (unsigned long long)n_full);
                    atomicAdd((unsigned long long *)&p.tile_stats[N * N + rr * N + cnt_d],
                              (unsigned long long)n_part);
                }
            }
            n_full = n_part = 0;
        };
        bool ok = mbar_wait_cl(bar(bars->kv_full), 0, p.wc) && issue_s(0) && issue_dp(0);
        for (int i = 0; i < nt && ok; ++i, piter_next(it, N, b, nq)) {
            // dV += P^T dO_i: P^T (bf16 pairs) in TMEM columns [0,32) for
            // queries 0..63 and [64,96) for 64..127; B = head-dim half of dO_i
            if (!mbar_wait_cl(bar(bars->p_ready), i & 1, p.wc)) break;
            if (!mbar_wait_cl(bar(bars->dov_full), i & 1, p.wc)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ts_pair(tdV, tS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                            sdesc_sw128(sbase + kOffDOV + kk * 2048, kBox, 1024), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit_pair(bar(bars->dov_empty));
            if (i + 1 < nt && !issue_s(i + 1)) break;
            // dQ_i = dS_i K over the pair's 256 keys (A = dSX, B = KQ; M = 128)
            if (!mbar_wait_cl(bar(bars->ds_ready), i & 1, p.wc)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_ss_pair(tdP, sdesc_sw128(sbase + kOffDSX + (kk >> 3) * kBox + (kk & 7) * 2048, kBox, 1024),
                            sdesc_sw128(sbase + kOffKQ + (kk >> 3) * kBox + (kk & 7) * 2048, kBox, 1024), id_q,
                            kk > 0 ? 1u : 0u);
            mma_commit_pair_mc(bar(bars->dq_full), kBothCtas);
            // dK += dS^T Q_i (A = own dS tile read K-major, B = head-dim half of Q_i)
            if (!mbar_wait_cl(bar(bars->qk_full), i & 1, p.wc)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss_pair(tdK, sdesc_sw128(sbase + kOffDS + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                            sdesc_sw128(sbase + kOffQK + kk * 2048, kBox, 1024), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit_pair(bar(bars->qk_empty));
            mma_commit_pair_mc(bar(bars->dk_done), kBothCtas);
            if (it.d != cnt_d) {
                flush_counts();
                cnt_d = it.d;
            }
            if (it.a == b) ++n_part;
            else ++n_full;
            if (i + 1 < nt) {
                if (!mbar_wait_cl(bar(bars->dq_free), i & 1, p.wc)) break;
                tc_fence_after();
                if (!issue_dp(i + 1)) break;
            }
        }
        flush_counts();
        if (ok) mma_commit_pair_mc(bar(bars->acc_done), kBothCtas);
        // every MMA issued above completes before tensor memory is freed
        mma_commit_pair(bar(bars->drain));
        mbar_wait_cl(bar(bars->drain), 0, p.wc);
    } else if (warp >= 4) {
        // ---------------- compute (both CTAs)
        const int wg = (warp - 4) >> 2;       // query columns [64 wg, 64 wg + 64)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // key row of S^T / dP^T
        const int cbase = wg * 64;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float cl2 = g.scale * 1.4426950408889634f;
        const uint32_t p_ready_cl = mapa_shared(bar(bars->p_ready), 0);
        const uint32_t ds_ready_cl = mapa_shared(bar(bars->ds_ready), 0);
        const uint32_t dq_free_cl = mapa_shared(bar(bars->dq_free), 0);
        // this row of dS^T: query half wg of the own tile, and the same values
        // into CTA wg's dSX (slot `rank`, this CTA's key tile)
        const uint32_t ds_own = sbase + kOffDS + wg * kBox + row * 128;
        const uint32_t ds_x = mapa_shared(sbase + kOffDSX + rank * kBox + row * 128, (uint32_t)wg);
        bool ok = nt > 0;

        auto stat_ptr = [&](int i) -> const float * {
            return reinterpret_cast<const float *>(smem + kOffStat + (i & 1) * kStatBytes) + cbase;
        };
        uint32_t pkP[32];  // P^T of the current tile (bf16 pairs), kept for dS
        auto compute_p = [&](const PairIter &t, int i) -> bool {
            if (!mbar_wait(bar(bars->st_full[i & 1]), (i >> 1) & 1, p.wc)) return false;
            if (!mbar_wait_cl(bar(bars->s_full), i & 1, p.wc)) return false;
            tc_fence_after();
            const float *sL = stat_ptr(i);
            // diagonal tile: keep (query col, key row) iff row <= col + [e <= d] - 1
            const int cmin = t.a == b ? row - ((e <= t.d) ? 0 : -1) : 0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t rr[32];
                tmem_ld32(tS + lane_off + cbase + c * 32, rr);
                tmem_ld_wait(rr);
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c0 = c * 32 + 2 * u;
                    const float p0 = ex2(fmaf(__uint_as_float(rr[2 * u]), cl2, -sL[c0]));
                    const float p1 = ex2(fmaf(__uint_as_float(rr[2 * u + 1]), cl2, -sL[c0 + 1]));
                    pk[u] = pack_bf16x2(cbase + c0 >= cmin ? p0 : 0.f, cbase + c0 + 1 >= cmin ? p1 : 0.f);
                    pkP[c * 16 + u] = pk[u];
                }
                tmem_st16(tS + lane_off + cbase + c * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cl(p_ready_cl);
            return true;
        };

        PairIter cur{0, 0, nq - 1};
        if (ok) ok = compute_p(cur, 0);
        for (int i = 0; i < nt && ok; ++i) {
            // ---- dS = P * (dP - Delta) -> own dS tile and the dSX of CTA wg
            if (!mbar_wait_cl(bar(bars->dp_full), i & 1, p.wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // this warp's rows of the own dS tile staged dQ_{i-1} for its bulk
            // reduction: that must have read them before they are overwritten
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
            const float *sD = stat_ptr(i) + 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t rr[32];
                tmem_ld32(tdP + lane_off + cbase + c * 32, rr);
                tmem_ld_wait(rr);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int u = v * 4 + h;
                        const int c0 = c * 32 + 2 * u;
                        __nv_bfloat162 pv = *reinterpret_cast<__nv_bfloat162 *>(&pkP[c * 16 + u]);
                        const float2 pf = __bfloat1622float2(pv);
                        w[h] = pack_bf16x2(pf.x * (__uint_as_float(rr[2 * u]) - sD[c0]),
                                           pf.y * (__uint_as_float(rr[2 * u + 1]) - sD[c0 + 1]));
                    }
                    const uint32_t sw = (uint32_t)(((c * 4 + v) ^ (row & 7)) * 16);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ds_own + sw), "r"(w[0]), "r"(w[1]),
                                 "r"(w[2]), "r"(w[3])
                                 : "memory");
                    st_cluster_v4(ds_x + sw, w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            fence_proxy_async_cluster();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_cl(ds_ready_cl);
                mbar_arrive(bar(bars->st_empty[i & 1]));  // tile i's statistics are done with
            }
            const PairIter done = cur;
            if (i + 1 < nt) {
                piter_next(cur, N, b, nq);
                if (!compute_p(cur, i + 1)) {
                    ok = false;
                    break;
                }
            }
            // ---- dQ_i: this CTA's 64 query rows (half `rank`); warp quarter q
            // reads TMEM lanes 32q..32q+31 = query rows 32(q&1)+lane of the
            // half, head-dimension block 64(q>>1); warpgroup wg takes columns
            // [32 wg, 32 wg + 32) of the block.  The 32 x 32 fp32 block goes to
            // the accumulator by a TMA bulk reduce-add (an asynchronous copy,
            // so the cluster-scope releases above never wait for it) from the
            // 4 KB of the own dS tile that this warp writes (free once dK_i
            // has read it).
            if (!mbar_wait_cl(bar(bars->dq_full), i & 1, p.wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t q0[32];
            tmem_ld32(tdP + lane_off + wg * 32, q0);
            tmem_ld_wait(q0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cl(dq_free_cl);
            if (!mbar_wait_cl(bar(bars->dk_done), i & 1, p.wc)) {
                ok = false;
                break;
            }
            const uint32_t stage = sbase + kOffDS + wg * kBox + quarter * 32 * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + lane * 128 + ((j ^ (lane & 7)) * 16)),
                             "r"(q0[4 * j]), "r"(q0[4 * j + 1]), "r"(q0[4 * j + 2]), "r"(q0[4 * j + 3])
                             : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int bq = (int)(bh * G + done.h);
                tma_reduce_add_4d(&tmdQ, stage, (quarter >> 1) * 64 + wg * 32,
                                  done.a * PT + 64 * (int)rank + (quarter & 1) * 32, done.d, bq);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group0();  // every reduction has landed
        if (ok) {
            ok = mbar_wait_cl(bar(bars->acc_done), 0, p.wc);
            tc_fence_after();
        }
        // ---------------- epilogue: this warpgroup's head-dim columns of dK, dV
        const int64_t kj = (int64_t)b * PT + row;
        const int64_t krow = bh * g.stride_bh + (int64_t)e * g.stripe_stride + kj * PT + cbase;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t tacc = which ? tdK : tdV;
            __nv_bfloat16 *outp = which ? p.dk : p.dv;
            const float mul = which ? g.scale : 1.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t rr[32];
                if (ok) {
                    tmem_ld32(tacc + lane_off + cbase + c * 32, rr);
                    tmem_ld_wait(rr);
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) rr[u] = 0u;
                }
                uint4 *dstp = reinterpret_cast<uint4 *>(outp + krow + c * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * mul, __uint_as_float(rr[8 * v + 1]) * mul);
                    w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * mul, __uint_as_float(rr[8 * v + 3]) * mul);
                    w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * mul, __uint_as_float(rr[8 * v + 5]) * mul);
                    w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * mul, __uint_as_float(rr[8 * v + 7]) * mul);
                    dstp[v] = w;
                }
            }
        }
    }
    // Neither CTA leaves (or frees tensor memory) while the other may still
    // arrive on its barriers or read its operands.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem, 512);
    }
    cluster_sync();
}

}  // namespace

// Striped placement, head dimension 128, whole 128-row tiles per stripe, an
// even number of stripes (key stripes e0, e0 + 1 pair up), dense batch.
bool bwd_pair_eligible(const AttnGeom &g) {
    return g.layout == STRIPED_LAYOUT_STRIPED && g.D == PT && g.seqs.n == 0 && g.N % 2 == 0 && g.L > 0 &&
           g.L % PT == 0;
}

int launch_tc_bwd_pair_main(const void *q, const void *k, const void *v, const void *dO, float *dq_acc,
                            const float *stats, void *dk, void *dv, const AttnGeom &g, int64_t *tile_stats,
                            cudaStream_t stream) {
    if (!bwd_pair_eligible(g)) return STRIPED_ERR_UNSUPPORTED;
    static PerDeviceOnce attr_once;
    const int attr = attr_once.get([] {
        return cuda_status(cudaFuncSetAttribute(tc_bwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kPairSmemBytes));
    });
    if (attr != STRIPED_OK) return attr;
    CUtensorMap mq, mqh, mk, mv, mdo, mdoh, mdq;
    const int64_t bh_kv = g.BH / g.G;
    int st;
    if ((st = make_bf16_map(&mq, q, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mqh, q, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 64)) ||
        (st = make_bf16_map(&mk, k, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mv, v, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mdo, dO, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mdoh, dO, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 64)) ||
        (st = make_f32_map(&mdq, dq_acc, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 32)))
        return st;
    PairParams p{};
    p.g = g;
    p.stats = stats;
    p.dq_acc = dq_acc;
    p.dk = (__nv_bfloat16 *)dk;
    p.dv = (__nv_bfloat16 *)dv;
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nclusters = (g.L / PT) * (g.N / 2) * bh_kv;
    if (2 * nclusters > 0x7fffffffll) return STRIPED_ERR_UNSUPPORTED;
    tc_bwd_pair_kernel<<<(unsigned)(2 * nclusters), kPairThreads, kPairSmemBytes, stream>>>(mq, mqh, mk, mv, mdo,
                                                                                            mdoh, mdq, p);
    return cuda_status(cudaGetLastError());
}

}  // namespace striped
