// attn_bwd_tc.cu -- bf16 striped causal attention backward on tcgen05.
//
// The pages use the method to train causal models (research.elamur.ai
// summary page, §Summary) but give no backward formulas; this is the
// derivative of the exact causal attention the forward computes.  With
// P = exp(scale q k^T - LSE) on kept pairs and Delta_p = <dO_p, O_p>:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),
//   dK = scale * dS^T Q,  dQ = scale * dS K.
// The same ring schedule and tile skipping as the forward: the key tile of
// stripe e is visited, in ring rounds r = 0..N-1, by the query stripe of
// device d = (e + r) mod N (the device that holds stripe e in round r).
//
// Three kernels:
//   bwd_pre    Delta_p = <dO_p, O_p> (fp32) and zero the fp32 dQ accumulator
//   bwd_main   one CTA per 128-key tile; loops over the query tiles that see
//              it (of every query head that reads its key/value head, with
//              grouped-query attention, and of its own sequence only, with
//              packed sequences).  warp 0 = TMA producer (K, V once; then
//              Q_i with its statistics, 2 stages), warp 2 = TMA producer of
//              dO_i (own 2-stage stream), warp 1 = TMEM allocator + MMA
//              issuer, warps 4..11 = two compute warpgroups; thread t of a
//              warpgroup owns key row t of S^T/dP^T and, for dQ_i, head-
//              dimension column t of its 64 queries (HD = 128) or query row
//              t (HD = 64); warpgroup 0 has query columns 0..63 and the
//              head-dimension columns 0..HD/2-1 of dK, dV (and of dQ at
//              HD = 64), warpgroup 1 the rest.  HD = 128 or 64.
//              TMEM: S^T [0,128) (P^T bf16 pairs over it), dP^T [128,256)
//              (dQ_i over it once dS_i is formed), dV [256,256+HD),
//              dK [256+HD,256+2HD).
//                S^T  = K Q_i^T      SS, both K-major
//                dP^T = V dO_i^T     SS, both K-major
//                dV  += P^T dO_i     TS, A = P^T in TMEM, B = dO_i MN-major
//                dK  += dS^T Q_i     SS, A = dS smem tile read K-major
//                dQ_i^T = K^T dS^T   SS, A = K read MN-major, B = the dS
//                                    tile read MN-major (HD = 128)
//                dQ_i = dS K         SS, A = the dS tile read MN-major (HD 64)
//              The dS tile ([key][query], 128-byte swizzle) is a valid
//              operand both ways, so dS^T never goes through TMEM.  Issue
//              order dV_i, S_{i+1}, dK_i, dQ_i, dP_{i+1} keeps the tensor core
//              busy while the compute warps form dS_i, P_{i+1} and read dQ_i
//              out; dK_i goes before dQ_i so that Q_i, whose last reader it
//              is, returns to the producer one MMA earlier and the next Q
//              tile loads early.
//              dQ_i to the fp32 accumulator: at HD = 128 dQ_i is formed
//              transposed (head dimension in TMEM lanes, queries in columns),
//              so a warp's reduction for one query covers one whole 128-byte
//              line of the accumulator, and dO_i returns to its producer as
//              soon as dV_i completes.  At HD = 64 (an M = 64 transposed
//              product would use another TMEM layout) warpgroup 0 adds its
//              columns with vector reductions and warpgroup 1 stages its
//              columns in the dO_i buffer, dead by then, and bulk
//              reduce-adds them (the wait for the reduce to read the buffer
//              is deferred by one tile).
//   bwd_post   dQ = bf16(scale * accumulator)
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace striped {

namespace {

constexpr int BT = 128;
constexpr int QS = 2;  // Q/dO stages
constexpr uint32_t kBox = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte-swizzle box)
constexpr uint32_t kStatBytes = 2 * 128 * 4;
constexpr int kThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 4..11 compute

// Shared-memory plan for head dimension HD (64 or 128): K, V, Q_i, dO_i
// tiles of HD/64 boxes; the dS tile is always 128 x 128.
template <int HD>
struct BwdCfg {
    static constexpr uint32_t kTile = (HD / 64) * kBox;
    static constexpr uint32_t kKOff = 0;
    static constexpr uint32_t kVOff = kTile;
    static constexpr uint32_t kQOff = 2 * kTile;                // stage s: Q at kQOff + s*2*kTile, dO after
    static constexpr uint32_t kDSOff = kQOff + QS * 2 * kTile;  // dS (MN-major A operand)
    static constexpr uint32_t kStatOff = kDSOff + 2 * kBox;     // per stage: [LSE*log2e 128 | Delta 128]
    static constexpr uint32_t kBarOff = kStatOff + QS * kStatBytes;
    static constexpr size_t kSmemBytes = kBarOff + 256;           // the dynamic smem base is 1024-aligned
    static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");
};

struct BwdParams {
    AttnGeom g;
    int d_fixed, e_fixed, first;  // one ring round only: query stripe, key stripe, start the dK/dV sums
    float *dk_acc, *dv_acc;       // one ring round only: fp32 dK, dV sums of the key block
    const float *stats;  // [BH][N][nq][LSE*log2e 128 | Delta 128], padded per 128-row tile
    float *dq_acc;       // [BH][S][D] fp32
    __nv_bfloat16 *dk, *dv;
    int64_t *tile_stats;
    WaitCtl wc;  // status word, wait bound, test hook
};

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[QS], q_empty[QS];    // Q_i + statistics of tile i
    uint64_t do_full[QS], do_empty[QS];  // dO_i (HD 64: its buffer also stages half of dQ_i)
    uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, acc_done;
    uint64_t drain;  // every MMA of the issuer has completed (before TMEM is freed)
    uint32_t tmem_slot;
};

__device__ __forceinline__ int tile_rows(int64_t L, int t) {
    const int64_t r = L - (int64_t)t * BT;
    return r >= BT ? BT : (int)r;
}

// Order in which a key tile visits its query tiles: the G query heads that
// read its key/value head (grouped-query attention; G = 1 otherwise), per
// head the query stripes d = 0, 1, ..., N-1, and within a stripe the tiles
// that see the key tile from the last one down (ascending order and ring
// order across the stripes measured within 2% of this one).
struct QTileIter {
    int h, k, d, a, a_lo, has_diag, diag_off;
};

__device__ __forceinline__ void qiter_seek(QTileIter &it, int layout, int N, int G, int e, int b, int nq,
                                           int rows_b, int dsel) {
    while (it.h < G) {
        while (it.k < N) {
            it.d = it.k;
            if (dsel >= 0 && it.d != dsel) {  // one ring round: only query stripe dsel
                ++it.k;
                continue;
            }
            const QuerySpan sp = query_span(layout, it.d, e, b, nq, rows_b);
            if (sp.a_lo < nq) {
                it.a_lo = sp.a_lo;
                it.has_diag = sp.has_diag;
                it.diag_off = sp.diag_off;
                it.a = nq - 1;
                return;
            }
            ++it.k;
        }
        it.k = 0;
        ++it.h;
    }
}

__device__ __forceinline__ QTileIter qiter_begin(int layout, int N, int G, int e, int b, int nq, int rows_b,
                                                 int dsel) {
    QTileIter it{0, 0, 0, 0, 0, 0, 0};
    qiter_seek(it, layout, N, G, e, b, nq, rows_b, dsel);
    return it;
}

__device__ __forceinline__ void qiter_next(QTileIter &it, int layout, int N, int G, int e, int b, int nq,
                                           int rows_b, int dsel) {
    if (--it.a < it.a_lo) {
        ++it.k;
        qiter_seek(it, layout, N, G, e, b, nq, rows_b, dsel);
    }
}


// kPacked: packed variable-length sequences (the sequence table is
// consulted); the dense instantiation compiles the span as {0, nq}.
// kRound: one ring round (ring_round_bwd): the key block of stripe e_fixed
// against the query block of stripe d_fixed, each its own [BH][L][D]
// tensor (stripe coordinate 0 in the tensor maps), dK and dV added into
// fp32 sums that travel with the key block.
template <int HD, bool kPacked, bool kRound = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
    using Cfg = BwdCfg<HD>;
    constexpr uint32_t kTile = Cfg::kTile, kKOff = Cfg::kKOff, kVOff = Cfg::kVOff, kQOff = Cfg::kQOff,
                       kDSOff = Cfg::kDSOff, kStatOff = Cfg::kStatOff;
    constexpr int kBoxes = HD / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    if ((smem_u32(smem) & 1023u) != 0) {  // operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) record_error(p.wc.st, STRIPED_ERR_ALIGN);
        return;
    }
    Bars *bars = reinterpret_cast<Bars *>(smem + Cfg::kBarOff);
    const uint32_t sbase = smem_u32(smem);
    const AttnGeom &g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int N = g.N;
    const int nq = (int)((g.L + BT - 1) / BT);

    // Head-major order: resident CTAs belong to one key/value head and sweep
    // its query tiles in the same order, sharing Q/dO tiles and dQ
    // accumulator lines in L2.  Within a head the heaviest key tiles (small
    // b) go first.  bh is the key/value head; query head bh*G + it.h.
    const int G = (int)g.G;
    const int64_t id = blockIdx.x;
    const int64_t per_head = kRound ? (int64_t)nq : (int64_t)nq * N;
    const int64_t bh = id / per_head;
    const int rem = (int)(id % per_head);
    const int bg = kRound ? rem : rem / N;  // key tile in the slice of stripe e
    const int e = kRound ? p.e_fixed : rem % N;
    const int dsel = kRound ? p.d_fixed : -1;  // one ring round: its query stripe only
    const int kst = kRound ? 0 : e;            // stripe coordinate of the key block in its tensor map
    const int rows_b = tile_rows(g.L, bg);
    // packed sequences: the key tile sees the query tiles of its own sequence
    // only (tiles qbase .. qbase + nqs - 1 of every slice)
    const SeqSpan sq = kPacked ? seq_of(g.seqs, bg, BT, nq) : SeqSpan{0, nq};
    const int b = bg - sq.start;  // key tile inside the sequence
    const int nqs = sq.count;
    const int qbase = sq.start;

    int nt = 0;
    for (int d = 0; d < N; ++d)
        if (dsel < 0 || d == dsel) nt += nqs - query_span(g.layout, d, e, b, nqs, rows_b).a_lo;
    nt *= G;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        for (int s = 0; s < QS; ++s) {
            mbar_init(smem_u32(&bars->q_full[s]), 1);
            mbar_init(smem_u32(&bars->q_empty[s]), 1);   // released by dK_i's commit
            mbar_init(smem_u32(&bars->do_full[s]), 1);
            mbar_init(smem_u32(&bars->do_empty[s]), HD == 128 ? 1 : 4);  // dV_i's commit; HD 64: warpgroup-1 warps
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->p_ready), 8);
        mbar_init(smem_u32(&bars->ds_ready), 8);
        mbar_init(smem_u32(&bars->dq_full), 1);
        mbar_init(smem_u32(&bars->dq_free), 8);
        mbar_init(smem_u32(&bars->acc_done), 1);
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
    const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + HD;

    if (warp == 0 && lane == 0 && nt > 0) {
        // ---------------- TMA producer: K, V once, then Q_i + statistics
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        const uint32_t kb = smem_u32(&bars->kv_full);
        mbar_arrive_expect_tx(kb, 2 * kTile);
#pragma unroll
        for (int x = 0; x < kBoxes; ++x) tma_load_4d(sbase + kKOff + x * kBox, &tmK, kb, 64 * x, bg * BT, kst, (int)bh);
#pragma unroll
        for (int x = 0; x < kBoxes; ++x) tma_load_4d(sbase + kVOff + x * kBox, &tmV, kb, 64 * x, bg * BT, kst, (int)bh);
        // test hook: the first Q tile is never loaded, so every wait on it
        // runs out (the kernel must then record the timeout and return)
        const bool skip_first = p.wc.inject == kInjectBwdSkipQ;
        QTileIter it = qiter_begin(g.layout, N, G, e, b, nqs, rows_b, dsel);
        int i = 0;
        for (; i < nt; ++i, qiter_next(it, g.layout, N, G, e, b, nqs, rows_b, dsel)) {
            const int s = i % QS;
            if (i >= QS && !mbar_wait(smem_u32(&bars->q_empty[s]), ((i / QS) + 1) & 1, p.wc)) break;
            if (skip_first && i == 0) continue;
            const uint32_t fb = smem_u32(&bars->q_full[s]);
            const uint32_t qdst = sbase + kQOff + s * 2 * kTile;
            const int64_t bq = bh * G + it.h;  // query head
            mbar_arrive_expect_tx(fb, kTile + kStatBytes);
            const int qst = kRound ? 0 : it.d;  // stripe coordinate of the query block
            bulk_load(sbase + kStatOff + s * kStatBytes,
                      p.stats + (((bq * (kRound ? 1 : N) + qst) * (int64_t)nq + qbase + it.a) << 8), kStatBytes, fb);
#pragma unroll
            for (int x = 0; x < kBoxes; ++x)
                tma_load_4d(qdst + x * kBox, &tmQ, fb, 64 * x, (qbase + it.a) * BT, qst, (int)bq);
        }
        // K, V and loads [0, i) were issued: wait (bounded) for the last of
        // each stage, so that on an error path none lands after the CTA exits
        mbar_wait(kb, 0, p.wc);
        for (int t = i > QS ? i - QS : 0; t < i; ++t)
            if (!(skip_first && t == 0)) mbar_wait(smem_u32(&bars->q_full[t % QS]), (t / QS) & 1, p.wc);
    } else if (warp == 2 && lane == 0 && nt > 0) {
        // ---------------- TMA producer: dO_i (its own stream: the buffer is
        // released at dV_i, or at HD 64 after the dQ_i half staged in it is read)
        tma_prefetch_desc(&tmdO);
        QTileIter it = qiter_begin(g.layout, N, G, e, b, nqs, rows_b, dsel);
        int i = 0;
        for (; i < nt; ++i, qiter_next(it, g.layout, N, G, e, b, nqs, rows_b, dsel)) {
            const int s = i % QS;
            if (i >= QS && !mbar_wait(smem_u32(&bars->do_empty[s]), ((i / QS) + 1) & 1, p.wc)) break;
            const uint32_t fb = smem_u32(&bars->do_full[s]);
            const uint32_t odst = sbase + kQOff + s * 2 * kTile + kTile;
            const int bq = (int)(bh * G + it.h);
            mbar_arrive_expect_tx(fb, kTile);
#pragma unroll
            for (int x = 0; x < kBoxes; ++x)
                tma_load_4d(odst + x * kBox, &tmdO, fb, 64 * x, (qbase + it.a) * BT, kRound ? 0 : it.d, bq);
        }
        for (int t = i > QS ? i - QS : 0; t < i; ++t)  // in-flight loads, as above
            mbar_wait(smem_u32(&bars->do_full[t % QS]), (t / QS) & 1, p.wc);
    } else if (warp == 1 && lane == 0 && nt > 0) {
        // ---------------- MMA issuer
        // Per query tile i (TMEM: S = S^T then P^T; DP = dP^T then dQ_i):
        //   dV += P^T dO | S(i+1) | dK += dS^T Q | dQ_i = dS K | dP(i+1)
        // so S(i+1) runs while the compute warps form dS_i and P(i+1), Q_i
        // is released at dK_i, and dP(i+1) follows as soon as dQ_i is out.
        constexpr uint32_t id_kk = idesc_bf16_f32(BT, BT, false, false);
        constexpr uint32_t id_kmn = idesc_bf16_f32(BT, HD, false, true);
        constexpr uint32_t id_mnmn = idesc_bf16_f32(BT, HD, true, true);
        constexpr uint32_t id_dqt = idesc_bf16_f32(HD, BT, true, true);  // dQ^T: M = HD, N = 128 queries
        auto issue_s = [&](int t) -> bool {
            const int s = t % QS;
            if (!mbar_wait(smem_u32(&bars->q_full[s]), (t / QS) & 1, p.wc)) return false;
            tc_fence_after();
            const uint32_t qaddr = sbase + kQOff + s * 2 * kTile;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                mma_ss(tS, sdesc_sw128(sbase + kKOff + off, 16, 1024), sdesc_sw128(qaddr + off, 16, 1024),
                       id_kk, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->s_full));
            return true;
        };
        auto issue_dp = [&](int t) -> bool {
            if (!mbar_wait(smem_u32(&bars->do_full[t % QS]), (t / QS) & 1, p.wc)) return false;
            tc_fence_after();
            const uint32_t oaddr = sbase + kQOff + (t % QS) * 2 * kTile + kTile;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                mma_ss(tdP, sdesc_sw128(sbase + kVOff + off, 16, 1024), sdesc_sw128(oaddr + off, 16, 1024),
                       id_kk, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->dp_full));
            return true;
        };
        // tiles whose five MMAs were issued, per query stripe: added to the
        // (round, device) counter when the stripe changes
        QTileIter it = qiter_begin(g.layout, N, G, e, b, nqs, rows_b, dsel);
        int cnt_d = -1, n_full = 0, n_part = 0;
        auto flush_counts = [&]() {
            if (p.tile_stats && cnt_d >= 0 && (n_full | n_part)) {
                const int rr = ring_round_of(cnt_d, e, N);
                atomicAdd((unsigned long long *)&p.tile_stats[rr * N + cnt_d], (unsigned long long)n_full);
                atomicAdd((unsigned long long *)&p.tile_stats[N * N + rr * N + cnt_d], (unsigned long long)n_part);
            }
            n_full = n_part = 0;
        };
        bool ok = mbar_wait(smem_u32(&bars->kv_full), 0, p.wc) && issue_s(0);
        if (ok) ok = issue_dp(0);
        for (int i = 0; i < nt && ok; ++i, qiter_next(it, g.layout, N, G, e, b, nqs, rows_b, dsel)) {
            const int s = i % QS;
            const uint32_t qaddr = sbase + kQOff + s * 2 * kTile;
            const uint32_t oaddr = qaddr + kTile;
            // dV += P^T dO: P^T (bf16 pairs) in TMEM columns [0,32) for
            // queries 0..63 and [64,96) for queries 64..127
            if (!mbar_wait(smem_u32(&bars->p_ready), i & 1, p.wc)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
                mma_ts(tdV, tS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                       sdesc_sw128(oaddr + kk * 2048, kBox, 1024), id_kmn, (i > 0 || kk > 0) ? 1u : 0u);
            // HD 128: dO_i (read by dP_i and dV_i only) is free once dV_i completes
            if (HD == 128 && i + QS < nt) mma_commit(smem_u32(&bars->do_empty[s]));
            if (i + 1 < nt && !issue_s(i + 1)) break;
            // dK += dS^T Q (A = dS^T, K-major view of the dS smem tile)
            if (!mbar_wait(smem_u32(&bars->ds_ready), i & 1, p.wc)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
                mma_ss(tdK, sdesc_sw128(sbase + kDSOff + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                       sdesc_sw128(qaddr + kk * 2048, kBox, 1024), id_kmn, (i > 0 || kk > 0) ? 1u : 0u);
            // Q_i (and its statistics) are free once dK_i completes
            if (i + QS < nt) mma_commit(smem_u32(&bars->q_empty[s]));
            if constexpr (HD == 128) {
                // dQ_i^T = K^T dS^T (A = K, MN-major; B = the dS tile, MN-major)
                // -> DP columns, head dimension in TMEM lanes, queries in columns
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk)
                    mma_ss(tdP, sdesc_sw128(sbase + kKOff + kk * 2048, kBox, 1024),
                           sdesc_sw128(sbase + kDSOff + kk * 2048, kBox, 1024), id_dqt, kk > 0 ? 1u : 0u);
            } else {
                // dQ_i = dS K (A = dS, MN-major view of the same tile) -> DP columns
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk)
                    mma_ss(tdP, sdesc_sw128(sbase + kDSOff + kk * 2048, kBox, 1024),
                           sdesc_sw128(sbase + kKOff + kk * 2048, kBox, 1024), id_mnmn, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->dq_full));
            if (it.d != cnt_d) {
                flush_counts();
                cnt_d = it.d;
            }
            if (it.has_diag && it.a == it.a_lo) ++n_part;
            else ++n_full;
            if (i + 1 < nt) {
                if (!mbar_wait(smem_u32(&bars->dq_free), i & 1, p.wc)) break;
                tc_fence_after();
                if (!issue_dp(i + 1)) break;
            }
        }
        flush_counts();
        if (ok) mma_commit(smem_u32(&bars->acc_done));
        // every MMA issued above completes before TMEM is freed (error paths)
        mma_commit(smem_u32(&bars->drain));
        mbar_wait(smem_u32(&bars->drain), 0, p.wc);
    } else if (warp >= 4) {
        // ---------------- compute: two warpgroups split the 128 query columns
        // of S^T/dP^T (64 each) and the HD columns of dQ_i, dK, dV (HD/2 each)
        const int wg = (warp - 4) >> 2;       // 0: first half, 1: second half
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // key row of S^T/dP^T; query row of dQ
        const int cbase = wg * 64;            // first query column of this warpgroup
        // first head-dimension column of this warpgroup (at HD = 128 the same
        // value as cbase, and written so for the compiler)
        const int dbase = HD == 128 ? cbase : wg * (HD / 2);
        const uint32_t pbase = wg * 64;       // TMEM columns of this warpgroup's P^T pairs
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float cl2 = g.scale * 1.4426950408889634f;
        const bool key_valid = row < rows_b;
        uint8_t *sDS = smem + kDSOff + wg * kBox + row * 128;
        bool ok = nt > 0;

        // per-query statistics of tile i (bulk-copied with Q_i/dO_i):
        // LSE*log2e (+inf past the stripe end, so P = 0 there) and Delta
        auto stat_ptr = [&](int i) -> const float * {
            return reinterpret_cast<const float *>(smem + kStatOff + (i % QS) * kStatBytes) + cbase;
        };
        // P^T of tile t (index i): kept in registers (bf16 pairs) for dS and
        // written to TMEM as the A operand of dV += P^T dO
        uint32_t pkP[32];
        auto compute_p = [&](const QTileIter &t, int i) -> bool {
            if (!mbar_wait(smem_u32(&bars->q_full[i % QS]), (i / QS) & 1, p.wc)) return false;
            if (!mbar_wait(smem_u32(&bars->s_full), i & 1, p.wc)) return false;
            tc_fence_after();
            const float *sL = stat_ptr(i);
            const bool diag = t.has_diag && t.a == t.a_lo;
            // keep pair (query col, key row) iff row <= col + diag_off
            const int cmin = diag ? row - t.diag_off : 0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t rr[32];
                tmem_ld32(tS + lane_off + cbase + c * 32, rr);
                tmem_ld_wait(rr);
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; u += 2) {
                    // four row statistics per 16-byte shared-memory load
                    const float4 l4 = *reinterpret_cast<const float4 *>(sL + c * 32 + 2 * u);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c0 = c * 32 + 2 * (u + h);
                        const float p0 = ex2(fmaf(__uint_as_float(rr[2 * (u + h)]), cl2, -lv[2 * h]));
                        const float p1 = ex2(fmaf(__uint_as_float(rr[2 * (u + h) + 1]), cl2, -lv[2 * h + 1]));
                        const bool k0 = key_valid && (cbase + c0 >= cmin);
                        const bool k1 = key_valid && (cbase + c0 + 1 >= cmin);
                        pk[u + h] = pack_bf16x2(k0 ? p0 : 0.f, k1 ? p1 : 0.f);
                        pkP[c * 16 + u + h] = pk[u + h];
                    }
                }
                tmem_st16(tS + lane_off + pbase + c * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready));
            return true;
        };

        QTileIter cur = qiter_begin(g.layout, N, G, e, b, nqs, rows_b, dsel);
        // warpgroup 1, lane 0: stage whose dQ bulk reduce still reads shared
        // memory (-1: none); the wait for it is deferred to the next tile
        int pending = -1;
        auto release_pending = [&]() {
            if (pending >= 0) {
                bulk_wait_group_read0();
                mbar_arrive(smem_u32(&bars->do_empty[pending]));
                pending = -1;
            }
        };
        if (ok) ok = compute_p(cur, 0);
        for (int i = 0; i < nt && ok; ++i) {
            // ---- dS = P * (dP - Delta) -> smem (A operand of dQ and dK)
            if (!mbar_wait(smem_u32(&bars->dp_full), i & 1, p.wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *sD = stat_ptr(i) + 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t rr[32];
                tmem_ld32(tdP + lane_off + cbase + c * 32, rr);
                tmem_ld_wait(rr);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w[4];
                    // the chunk's eight Delta values in two 16-byte loads
                    const float4 d0 = *reinterpret_cast<const float4 *>(sD + c * 32 + 8 * v);
                    const float4 d1 = *reinterpret_cast<const float4 *>(sD + c * 32 + 8 * v + 4);
                    const uint64_t dd[4] = {f2(d0.x, d0.y), f2(d0.z, d0.w), f2(d1.x, d1.y), f2(d1.z, d1.w)};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int u = v * 4 + h;  // pair index within the chunk
                        __nv_bfloat162 pv = *reinterpret_cast<__nv_bfloat162 *>(&pkP[c * 16 + u]);
                        const float2 pf = __bfloat1622float2(pv);
                        // dS = P * (dP - Delta), two at a time
                        const float2 ds = f2_split(mul2(f2(pf.x, pf.y), sub2(f2(__uint_as_float(rr[2 * u]),
                                                                                  __uint_as_float(rr[2 * u + 1])), dd[h])));
                        w[h] = pack_bf16x2(ds.x, ds.y);
                    }
                    const int chunk = c * 4 + v;
                    *reinterpret_cast<uint4 *>(sDS + ((chunk ^ (row & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
            // the previous tile's dQ reduce has had dS_i's time to read its
            // staging: return that dO buffer to the producer now
            if (wg == 1 && lane == 0) release_pending();
            // ---- P of the next tile while the tensor core runs dQ_i / dK_i
            const QTileIter done = cur;
            if (i + 1 < nt) {
                qiter_next(cur, g.layout, N, G, e, b, nqs, rows_b, dsel);
                if (!compute_p(cur, i + 1)) {
                    ok = false;
                    break;
                }
            }
            // ---- dQ_i readout -> fp32 accumulator
            if (!mbar_wait(smem_u32(&bars->dq_full), i & 1, p.wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // dQ_i -> fp32 accumulator (the two forms are described at the
            // top of this file).
            const int s = i % QS;
            const int64_t bq = bh * G + done.h;  // query head of tile i
            if constexpr (HD == 128) {
                // dQ_i^T: lane = head-dimension column, TMEM column = query;
                // this warp's 32 dimensions of the warpgroup's 64 queries.
                // One reduction per query covers a whole 128-byte line of the
                // accumulator across the warp.
                uint32_t q0[32], q1[32];
                tmem_ld32(tdP + lane_off + cbase, q0);
                tmem_ld32(tdP + lane_off + cbase + 32, q1);
                tmem_ld_wait(q0);
                tmem_ld_wait(q1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
                const int64_t q_first = (int64_t)(qbase + done.a) * BT + cbase;
                const int64_t nv = g.L - q_first;  // real queries among the 64 (uniform per warp)
                float *dst = p.dq_acc +
                             (bq * g.stride_bh + (int64_t)done.d * g.stripe_stride + q_first * HD + quarter * 32 + lane);
                if (nv >= 64) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) red_add_f32(dst + c * HD, __uint_as_float(q0[c]));
#pragma unroll
                    for (int c = 0; c < 32; ++c) red_add_f32(dst + (32 + c) * HD, __uint_as_float(q1[c]));
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c < nv) red_add_f32(dst + c * HD, __uint_as_float(q0[c]));
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (32 + c < nv) red_add_f32(dst + (32 + c) * HD, __uint_as_float(q1[c]));
                }
            } else {
                // HD = 64: split over two paths so neither the TMA engine nor
                // the load/store unit carries all of it: warpgroup 0 adds its 32
                // columns with vector reductions; warpgroup 1 stages its 32
                // columns in the dO_i buffer (dead once dV_i, covered by
                // dq_full, is done) as one 128-byte-swizzled box and each warp
                // bulk-reduces its own 32 rows, then returns the buffer.
                uint32_t q0[32];
                tmem_ld32(tdP + lane_off + dbase, q0);
                tmem_ld_wait(q0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
                if (wg == 0) {
                    const int64_t qi = (int64_t)(qbase + done.a) * BT + row;
                    if (qi < g.L) {
                        float *dst =
                            p.dq_acc + (bq * g.stride_bh + (int64_t)done.d * g.stripe_stride + qi * HD + dbase);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            red_add_v4(dst + 4 * v, __uint_as_float(q0[4 * v]), __uint_as_float(q0[4 * v + 1]),
                                       __uint_as_float(q0[4 * v + 2]), __uint_as_float(q0[4 * v + 3]));
                    }
                } else {
                    const uint32_t stage = sbase + kQOff + s * 2 * kTile + kTile;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t addr = stage + row * 128 + ((j ^ (row & 7)) * 16);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(q0[4 * j]),
                                     "r"(q0[4 * j + 1]), "r"(q0[4 * j + 2]), "r"(q0[4 * j + 3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t wofs = (uint32_t)quarter * 32 * 128;
                        const int r0 = (qbase + done.a) * BT + quarter * 32;
                        tma_reduce_add_4d(&tmdQ, stage + wofs, dbase, r0, kRound ? 0 : done.d, (int)bq);
                        bulk_commit_group();
                        pending = s;
                    }
                }
            }
        }
        if (wg == 1 && lane == 0) release_pending();
        if (lane == 0) bulk_wait_group0();
        if (ok) {
            ok = mbar_wait(smem_u32(&bars->acc_done), 0, p.wc);
            tc_fence_after();
        }
        // ---------------- epilogue: this warpgroup's columns of dK, dV
        const int64_t kj = (int64_t)bg * BT + row;
        const int64_t krow = bh * g.stride_bh + (int64_t)e * g.stripe_stride + kj * HD + dbase;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t tacc = which ? tdK : tdV;
            __nv_bfloat16 *outp = which ? p.dk : p.dv;
            const float mul = which ? g.scale : 1.f;
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                uint32_t rr[32];
                if (ok) {
                    tmem_ld32(tacc + lane_off + dbase + c * 32, rr);
                    tmem_ld_wait(rr);
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) rr[u] = 0u;
                }
                if (kRound && kj < g.L) {
                    // one ring round: add into (or, first, start) the block's fp32 sums
                    float *acc = (which ? p.dk_acc : p.dv_acc) + krow + c * 32;
#pragma unroll
                    for (int u = 0; u < 32; u += 4) {
                        float4 a4 = p.first ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<float4 *>(acc + u);
                        a4.x += __uint_as_float(rr[u]) * mul;
                        a4.y += __uint_as_float(rr[u + 1]) * mul;
                        a4.z += __uint_as_float(rr[u + 2]) * mul;
                        a4.w += __uint_as_float(rr[u + 3]) * mul;
                        *reinterpret_cast<float4 *>(acc + u) = a4;
                    }
                } else if (kj < g.L) {
                    uint4 *dst = reinterpret_cast<uint4 *>(outp + krow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * mul, __uint_as_float(rr[8 * v + 1]) * mul);
                        w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * mul, __uint_as_float(rr[8 * v + 3]) * mul);
                        w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * mul, __uint_as_float(rr[8 * v + 5]) * mul);
                        w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * mul, __uint_as_float(rr[8 * v + 7]) * mul);
                        dst[v] = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// Per row of every stripe, padded to whole 128-row tiles: the tile-major
// statistics block [LSE*log2e 128 | Delta 128] with Delta_p = <dO_p, O_p>
// (fp32); padding rows get LSE = +inf and Delta = 0.  Real rows also get
// their dQ accumulator row zeroed.  One warp per padded row; each lane
// covers HD/32 consecutive elements of it.
template <int HD>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      const float *__restrict__ lse, float *__restrict__ stats,
                                                      float *__restrict__ dq_acc, int64_t L, int nq,
                                                      int64_t padded_rows) {
    const int lane = threadIdx.x & 31;
    const int64_t per_stripe = (int64_t)nq * BT;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t pr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < padded_rows;
         pr += nwarps) {
        const int64_t stripe = pr / per_stripe;  // bh * N + d
        const int64_t ii = pr - stripe * per_stripe;
        float *blk = stats + ((stripe * nq + (ii >> 7)) << 8) + (ii & 127);
        if (ii >= L) {
            if (lane == 0) {
                blk[0] = INFINITY;
                blk[128] = 0.f;
            }
            continue;
        }
        const int64_t rw = stripe * L + ii;  // row of the [BH][S] tensors
        float sum;
        if constexpr (HD == 128) {
            const uint2 ov = *reinterpret_cast<const uint2 *>(o + rw * HD + lane * 4);
            const uint2 gv = *reinterpret_cast<const uint2 *>(dO + rw * HD + lane * 4);
            const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv);
            const float2 a0 = __bfloat1622float2(o2[0]), a1 = __bfloat1622float2(o2[1]);
            const float2 b0 = __bfloat1622float2(g2[0]), b1 = __bfloat1622float2(g2[1]);
            sum = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
        } else {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(o + rw * HD + lane * 2));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(dO + rw * HD + lane * 2));
            sum = a.x * b.x + a.y * b.y;
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) {
            blk[0] = lse[rw] * 1.4426950408889634f;
            blk[128] = sum;
        }
        if constexpr (HD == 128)
            *reinterpret_cast<float4 *>(dq_acc + rw * HD + lane * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        else
            *reinterpret_cast<float2 *>(dq_acc + rw * HD + lane * 2) = make_float2(0.f, 0.f);
    }
}

// dQ = bf16(scale * accumulator), 8 elements per thread per step.
__global__ void __launch_bounds__(256) bwd_post_kernel(const float *__restrict__ dq_acc,
                                                       __nv_bfloat16 *__restrict__ dq, int64_t n8, float scale) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += stride) {
        const float4 x = reinterpret_cast<const float4 *>(dq_acc)[2 * t];
        const float4 y = reinterpret_cast<const float4 *>(dq_acc)[2 * t + 1];
        uint4 w;
        w.x = pack_bf16x2(x.x * scale, x.y * scale);
        w.y = pack_bf16x2(x.z * scale, x.w * scale);
        w.z = pack_bf16x2(y.x * scale, y.y * scale);
        w.w = pack_bf16x2(y.z * scale, y.w * scale);
        reinterpret_cast<uint4 *>(dq)[t] = w;
    }
}

}  // namespace

int device_sm_count() {
    static PerDeviceOnce once;
    return once.get([] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        return n;
    });
}

namespace {

template <int HD>
int launch_bwd_hd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                  void *dq, void *dk, void *dv, float *dq_acc, float *stats, const AttnGeom &g, int64_t *tile_stats,
                  cudaStream_t stream) {
    constexpr size_t kSmemBytes = BwdCfg<HD>::kSmemBytes;
    static PerDeviceOnce attr_once;
    const int attr = attr_once.get([] {
        cudaError_t e = cudaFuncSetAttribute(tc_bwd_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_bwd_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_bwd_kernel<HD, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        return cuda_status(e);
    });
    if (attr != STRIPED_OK) return attr;
    const int64_t rows = g.BH * g.N * g.L;
    const int sms = device_sm_count();
    const int nq = (int)((g.L + BT - 1) / BT);
    bwd_pre_kernel<HD><<<sms * 8, 256, 0, stream>>>((const __nv_bfloat16 *)o, (const __nv_bfloat16 *)dO, lse,
                                                    stats, dq_acc, g.L, nq, g.BH * g.N * (int64_t)nq * BT);
    int st = cuda_status(cudaGetLastError());
    if (st != STRIPED_OK) return st;
    CUtensorMap mq, mk, mv, mdo;
    const int64_t bh_kv = g.BH / g.G;
    if ((st = make_bf16_map(&mq, q, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mk, k, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mv, v, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mdo, dO, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 128)))
        return st;
    CUtensorMap mdq;  // the dQ bulk reduce (read at HD = 64 only)
    if ((st = make_f32_map(&mdq, dq_acc, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 32))) return st;
    BwdParams p{};
    p.g = g;
    p.stats = stats;
    p.dq_acc = dq_acc;
    p.dk = (__nv_bfloat16 *)dk;
    p.dv = (__nv_bfloat16 *)dv;
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nk = (g.L + BT - 1) / BT;
    const int64_t nblocks = nk * g.N * bh_kv;  // one CTA per key tile of every key/value head
    if (nblocks > 0x7fffffffll) return STRIPED_ERR_UNSUPPORTED;
    if (g.seqs.n > 0)
        tc_bwd_kernel<HD, true><<<(unsigned)nblocks, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, p);
    else
        tc_bwd_kernel<HD, false><<<(unsigned)nblocks, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, p);
    st = cuda_status(cudaGetLastError());
    if (st != STRIPED_OK) return st;
    bwd_post_kernel<<<sms * 8, 256, 0, stream>>>(dq_acc, (__nv_bfloat16 *)dq, rows * HD / 8, g.scale);
    return cuda_status(cudaGetLastError());
}

template <int HD>
int launch_round_bwd_hd(const void *q_d, const void *k_e, const void *v_e, const void *dO_d, const float *stats,
                        float *dq_acc, float *dk_acc, float *dv_acc, int d, int e, int first, const AttnGeom &g,
                        int64_t *tile_stats, cudaStream_t stream) {
    constexpr size_t kSmemBytes = BwdCfg<HD>::kSmemBytes;
    static PerDeviceOnce attr_once;
    const int attr = attr_once.get([] {
        return cuda_status(cudaFuncSetAttribute(tc_bwd_kernel<HD, false, true>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
    });
    if (attr != STRIPED_OK) return attr;
    // every block is its own [BH][L][D] tensor: a stripe dimension of extent 1
    const int64_t ld = g.L * g.D;
    CUtensorMap mq, mk, mv, mdo, mdq;
    int st;
    if ((st = make_bf16_map(&mq, q_d, g.D, g.L, 1, g.BH, ld, ld, 128)) ||
        (st = make_bf16_map(&mk, k_e, g.D, g.L, 1, g.BH, ld, ld, 128)) ||
        (st = make_bf16_map(&mv, v_e, g.D, g.L, 1, g.BH, ld, ld, 128)) ||
        (st = make_bf16_map(&mdo, dO_d, g.D, g.L, 1, g.BH, ld, ld, 128)) ||
        (st = make_f32_map(&mdq, dq_acc, g.D, g.L, 1, g.BH, ld, ld, 32)))
        return st;
    BwdParams p{};
    p.g = g;
    p.g.G = 1;
    p.g.stride_bh = ld;
    p.g.stripe_stride = 0;
    p.d_fixed = d;
    p.e_fixed = e;
    p.first = first;
    p.dk_acc = dk_acc;
    p.dv_acc = dv_acc;
    p.stats = stats;
    p.dq_acc = dq_acc;
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nq = (g.L + BT - 1) / BT;
    const int64_t nblocks = nq * g.BH;
    if (nblocks > 0x7fffffffll) return STRIPED_ERR_UNSUPPORTED;
    tc_bwd_kernel<HD, false, true><<<(unsigned)nblocks, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, p);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_round_bwd_prepare(const void *o_d, const float *lse_d, const void *dO_d, float *stats, float *dq_acc,
                             const AttnGeom &g, cudaStream_t stream) {
    const int nq = (int)((g.L + BT - 1) / BT);
    const int sms = device_sm_count();
    const int64_t padded = g.BH * (int64_t)nq * BT;
    if (g.D == 64)
        bwd_pre_kernel<64><<<sms * 8, 256, 0, stream>>>((const __nv_bfloat16 *)o_d, (const __nv_bfloat16 *)dO_d,
                                                        lse_d, stats, dq_acc, g.L, nq, padded);
    else
        bwd_pre_kernel<128><<<sms * 8, 256, 0, stream>>>((const __nv_bfloat16 *)o_d, (const __nv_bfloat16 *)dO_d,
                                                         lse_d, stats, dq_acc, g.L, nq, padded);
    return cuda_status(cudaGetLastError());
}

int launch_tc_round_bwd(const void *q_d, const void *k_e, const void *v_e, const void *dO_d, const float *stats,
                        float *dq_acc, float *dk_acc, float *dv_acc, int d, int e, int first, const AttnGeom &g,
                        int64_t *tile_stats, cudaStream_t stream) {
    if (g.D == 64)
        return launch_round_bwd_hd<64>(q_d, k_e, v_e, dO_d, stats, dq_acc, dk_acc, dv_acc, d, e, first, g, tile_stats,
                                       stream);
    return launch_round_bwd_hd<128>(q_d, k_e, v_e, dO_d, stats, dq_acc, dk_acc, dv_acc, d, e, first, g, tile_stats,
                                    stream);
}

int launch_scale_to_bf16(const float *acc, void *out, int64_t n8, float mul, cudaStream_t stream) {
    bwd_post_kernel<<<device_sm_count() * 8, 256, 0, stream>>>(acc, (__nv_bfloat16 *)out, n8, mul);
    return cuda_status(cudaGetLastError());
}

int launch_tc_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dO, void *dq, void *dk, void *dv, float *dq_acc, float *stats,
                  const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream) {
    if (g.D == 64)
        return launch_bwd_hd<64>(q, k, v, o, lse, dO, dq, dk, dv, dq_acc, stats, g, tile_stats, stream);
    return launch_bwd_hd<128>(q, k, v, o, lse, dO, dq, dk, dv, dq_acc, stats, g, tile_stats, stream);
}

}  // namespace striped
