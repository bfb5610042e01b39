// attn_fwd_pair.cu -- bf16 striped causal attention forward, two query tiles
// per CTA whose softmax groups alternate on the tensor core.
//
// In the striped placement the query tiles of index a of stripes d and d+1
// visit the same key tiles in every ring round: tiles 0..a of key stripe e,
// tile a being the diagonal one, whose mask keeps j <= i when e <= d and
// j < i otherwise (research.elamur.ai summary page, §Summary: every device
// keeps about half of every round).  So one CTA runs both query tiles on one
// K/V stream.  Each query tile has its own softmax group, S buffer and O
// accumulator; the single MMA thread issues, per key tile j,
//     PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so that while one group turns S into P the tensor core works for the
// other group.  Used for the batched striped forward when every stripe is a
// whole number of tiles, N is even, the head dimension is 64 or 128 and the
// grid stays balanced (fwd_pair_eligible); the one-tile kernel serves every
// other case.
//
//   warp 0      TMA producer: Q_A, Q_B once, then K/V tiles (2 stages at
//               HD = 128, 4 at HD = 64)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  softmax group A (stripe d), thread t owns query row t
//   warps 6..9  softmax group B (stripe d + 1)
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+HD),
// O_B [384,384+HD); P is written back over S as bf16 pairs.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace striped {

namespace {

constexpr int PB = 128;                         // tile edge (queries and keys)
constexpr uint32_t kPBox = 128 * 128;           // 128 rows x 64 bf16
constexpr int kPMaxNS = 4;

// Shared-memory plan for head dimension HD (64 or 128): Q_A, Q_B, then PNS
// stages of K and V, each tile HD/64 boxes.
template <int HD>
struct PairCfg {
    static constexpr int PNS = HD == 128 ? 2 : 4;      // K/V stages
    static constexpr uint32_t kPTile = (HD / 64) * kPBox;  // 128 x HD bf16
    static constexpr uint32_t kPQOff = 0;                 // Q_A, then Q_B
    static constexpr uint32_t kPKVOff = 2 * kPTile;       // stage s: K at kPKVOff + s*kPStage, V after
    static constexpr uint32_t kPStage = 2 * kPTile;
    static constexpr uint32_t kPBarOff = kPKVOff + PNS * kPStage;
    static constexpr size_t kPSmemBytes = 1024 + kPBarOff + 256;
    static_assert(kPSmemBytes <= 232448, "shared memory over the per-block limit");
    static_assert(PNS <= kPMaxNS, "barrier array");
};
constexpr int kPThreads = 320;
constexpr float kPRescale = 8.0f;  // lazy rescale threshold, log2 units

struct PairBars {
    uint64_t q_full;
    uint64_t kv_full[kPMaxNS], kv_empty[kPMaxNS];
    uint64_t s_full[2], p_ready[2], o_done[2];  // per softmax group
    uint64_t drain;                             // every MMA of the issuer has completed
    uint32_t tmem_slot;
};

struct PairParams {
    AttnGeom g;
    __nv_bfloat16 *o;
    float *lse;
    int64_t *tile_stats;
    WaitCtl wc;  // status word, wait bound, test hook
};

template <int HD>
__global__ void __launch_bounds__(kPThreads, 1)
    tc_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PairParams p) {
    using Cfg = PairCfg<HD>;
    constexpr int PNS = Cfg::PNS;
    constexpr uint32_t kPTile = Cfg::kPTile, kPQOff = Cfg::kPQOff, kPKVOff = Cfg::kPKVOff,
                       kPStage = Cfg::kPStage, kPBarOff = Cfg::kPBarOff;
    constexpr int kBoxes = HD / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    PairBars *bars = reinterpret_cast<PairBars *>(smem + kPBarOff);
    const uint32_t sbase = smem_u32(smem);
    const AttnGeom &g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int N = g.N;
    const int nq = (int)(g.L / PB);  // whole tiles (checked by the launcher)
    const int npair = N / 2;

    // Head-major order, heaviest query tiles first (as the one-tile kernel).
    const int64_t id = blockIdx.x;
    const int64_t per_head = (int64_t)nq * npair;
    const int64_t bh = id / per_head;
    const int rem = (int)(id % per_head);
    const int a = nq - 1 - rem / npair;
    const int d0 = 2 * (rem % npair);  // group A: stripe d0, group B: stripe d0 + 1
    const int kvh = (int)(bh / g.G);
    const int ntr = a + 1;  // key tiles 0..a of every key stripe
    const int nt = N * ntr;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int s = 0; s < PNS; ++s) {
            mbar_init(smem_u32(&bars->kv_full[s]), 1);
            mbar_init(smem_u32(&bars->kv_empty[s]), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&bars->s_full[x]), 1);
            mbar_init(smem_u32(&bars->p_ready[x]), 4);
            mbar_init(smem_u32(&bars->o_done[x]), 1);
        }
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

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const uint32_t qb = smem_u32(&bars->q_full);
        mbar_arrive_expect_tx(qb, 2 * kPTile);
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int c = 0; c < kBoxes; ++c)
                tma_load_4d(sbase + kPQOff + x * kPTile + c * kPBox, &tmQ, qb, 64 * c, a * PB, d0 + x, (int)bh);
        // test hook: the first K/V tile is never loaded, so every wait on it
        // runs out (the kernel must then record the timeout and return)
        const bool skip_first = p.wc.inject == kInjectFwdSkipKV;
        int j = 0;
        for (int e = 0; e < N; ++e) {
            bool ok = true;
            for (int b = 0; b < ntr; ++b, ++j) {
                const int s = j % PNS;
                if (j >= PNS && !mbar_wait(smem_u32(&bars->kv_empty[s]), ((j / PNS) + 1) & 1, p.wc)) {
                    ok = false;
                    break;
                }
                if (skip_first && j == 0) continue;
                const uint32_t fb = smem_u32(&bars->kv_full[s]);
                const uint32_t kdst = sbase + kPKVOff + s * kPStage;
                const uint32_t vdst = kdst + kPTile;
                mbar_arrive_expect_tx(fb, 2 * kPTile);
#pragma unroll
                for (int c = 0; c < kBoxes; ++c) {
                    tma_load_4d(kdst + c * kPBox, &tmK, fb, 64 * c, b * PB, e, kvh);
                    tma_load_4d(vdst + c * kPBox, &tmV, fb, 64 * c, b * PB, e, kvh);
                }
            }
            if (!ok) break;
        }
        // loads [0, j) and Q were issued: wait (bounded) for the last of each
        // stage, so that on an error path none lands after the CTA has exited
        mbar_wait(qb, 0, p.wc);
        for (int t = j > PNS ? j - PNS : 0; t < j; ++t)
            if (!(skip_first && t == 0)) mbar_wait(smem_u32(&bars->kv_full[t % PNS]), (t / PNS) & 1, p.wc);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
        constexpr uint32_t idesc_qk = idesc_bf16_f32(PB, PB, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(PB, HD, false, true);
        bool ok = mbar_wait(smem_u32(&bars->q_full), 0, p.wc);
        tc_fence_after();
        auto issue_s = [&](int x, int t) -> bool {
            const int s = t % PNS;
            if (!mbar_wait(smem_u32(&bars->kv_full[s]), (t / PNS) & 1, p.wc)) return false;
            tc_fence_after();
            const uint32_t qaddr = sbase + kPQOff + x * kPTile;
            const uint32_t kaddr = sbase + kPKVOff + s * kPStage;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kPBox + (kk & 3) * 32;
                mma_ss(tmem + 128 * x, sdesc_sw128(qaddr + off, 16, 1024), sdesc_sw128(kaddr + off, 16, 1024),
                       idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->s_full[x]));
            return true;
        };
        auto issue_pv = [&](int x, int t) -> bool {
            if (!mbar_wait(smem_u32(&bars->p_ready[x]), t & 1, p.wc)) return false;
            tc_fence_after();
            const uint32_t vaddr = sbase + kPKVOff + (t % PNS) * kPStage + kPTile;
#pragma unroll
            for (int kk = 0; kk < PB / 16; ++kk)
                mma_ts(tmem + 256 + 128 * x, tmem + 128 * x + kk * 8, sdesc_sw128(vaddr + kk * 2048, kPBox, 1024),
                       idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&bars->o_done[x]));
            return true;
        };
        if (ok) ok = issue_s(0, 0) && issue_s(1, 0);
        for (int j = 0; j < nt && ok; ++j) {
            if (!issue_pv(0, j)) break;
            if (j + 1 < nt && !issue_s(0, j + 1)) break;
            if (!issue_pv(1, j)) break;
            // only stages the producer will refill get a release
            if (j + PNS < nt) mma_commit(smem_u32(&bars->kv_empty[j % PNS]));
            if (j + 1 < nt && !issue_s(1, j + 1)) break;
        }
        // every MMA issued above completes before TMEM is freed (error paths)
        mma_commit(smem_u32(&bars->drain));
        mbar_wait(smem_u32(&bars->drain), 0, p.wc);
    } else if (warp >= 2) {
        // ---------------- softmax + epilogue of one query tile
        const int x = (warp - 2) >> 2;       // group: 0 (stripe d0) or 1 (stripe d0 + 1)
        const int d = d0 + x;
        const int quarter = warp & 3;
        const int ri = quarter * 32 + lane;  // query row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + 128 * x + lane_off, tO = tmem + 256 + 128 * x + lane_off;
        const float cl2 = g.scale * 1.4426950408889634f;
        float m_ref = -INFINITY, l = 0.f;
        int j = 0;
        bool ok = true;
        for (int e = 0; e < N && ok; ++e) {
            // key tiles 0 .. nfull-1 in full, tile nfull (= a) under the
            // striped diagonal mask: keep key column <= row + diag_off
            const RoundSpan sp = round_span(STRIPED_LAYOUT_STRIPED, d, e, a, nq, PB);
            const int lim_diag = ri + sp.diag_off;
            int n_full = 0, n_part = 0;  // tiles of this round turned into P below
            for (int b = 0; b < ntr; ++b, ++j) {
                if (!mbar_wait(smem_u32(&bars->s_full[x]), j & 1, p.wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float sv[PB];
                {
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
                const bool diag = b == sp.nfull;
                if (diag) {
#pragma unroll
                    for (int c = 0; c < PB; ++c)
                        if (c > lim_diag) sv[c] = -INFINITY;
                }
                float mx8[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) mx8[t] = sv[t];
#pragma unroll
                for (int c = 8; c < PB; c += 16)
#pragma unroll
                    for (int t = 0; t < 8; ++t) mx8[t] = fmax3(mx8[t], sv[c + t], sv[c + 8 + t]);
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float m_tile = mx * cl2;
                const bool move = (j == 0) ? true : (m_tile > m_ref + kPRescale);
                const float m_new = move ? fmaxf(m_ref, m_tile) : m_ref;
                const float alpha = (j == 0 || !move) ? 1.f : ex2(m_ref - m_new);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                // P in two halves of 64 columns, each stored as soon as it is
                // packed (ten warps leave 168 registers a thread)
                // the same arithmetic, in the same order, as the one-tile
                // kernel (paired FMA for the exponent arguments, four paired
                // row-sum accumulators), so both give identical results
                const uint64_t cl2x2 = f2(cl2, cl2), nm2 = f2(-m_use, -m_use);
                uint64_t acc4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float2 x = f2_split(fma2(f2(sv[64 * h + 2 * c], sv[64 * h + 2 * c + 1]), cl2x2, nm2));
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        acc4[c & 3] = add2(acc4[c & 3], f2(p0, p1));
                        pk[c] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + 32 * h, pk);
                }
                const float2 s01 = f2_split(add2(acc4[0], acc4[1])), s23 = f2_split(add2(acc4[2], acc4[3]));
                const float sum = (s01.x + s01.y) + (s23.x + s23.y);
                tmem_st_wait();
                l = l * alpha + sum;
                m_ref = m_new;
                if (j > 0) {
                    // PV(j-1) of this group must be complete before O is touched
                    if (!mbar_wait(smem_u32(&bars->o_done[x]), (j - 1) & 1, p.wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
                        // rare (lazy rescale): one 32-column chunk at a time
                        // keeps the softmax thread within its registers
#pragma unroll 1
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t rr[32];
                            tmem_ld32(tO + c * 32, rr);
                            tmem_ld_wait(rr);
#pragma unroll
                            for (int u = 0; u < 32; ++u)
                                rr[u] = __float_as_uint(__uint_as_float(rr[u]) * alpha);
                            tmem_st32(tO + c * 32, rr);
                        }
                        tmem_st_wait();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready[x]));
                if (diag) ++n_part;
                else ++n_full;
            }
            // the round's counters get the tiles that ran (one thread a group)
            if (p.tile_stats && quarter == 2 && lane == 0 && (n_full | n_part)) {
                const int rr = ring_round_of(d, e, N);
                atomicAdd((unsigned long long *)&p.tile_stats[rr * N + d], (unsigned long long)n_full);
                atomicAdd((unsigned long long *)&p.tile_stats[N * N + rr * N + d], (unsigned long long)n_part);
            }
        }
        // ---------------- epilogue
        if (ok) {
            ok = mbar_wait(smem_u32(&bars->o_done[x]), (nt - 1) & 1, p.wc);
            tc_fence_after();
        }
        const int64_t i = (int64_t)a * PB + ri;
        const bool empty = !(l > 0.f) || !ok;
        const float inv_l = empty ? 0.f : 1.f / l;
        const float lse_row = empty ? -INFINITY : (m_ref + log2f(l)) * 0.6931471805599453f;
        p.lse[bh * g.lse_stride_bh + (int64_t)d * g.lse_stripe_stride + i] = lse_row;
        const int64_t orow = (int64_t)bh * g.stride_bh + (int64_t)d * g.stripe_stride + i * HD;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tO + c * 32, rr);
            tmem_ld_wait(rr);
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

}  // namespace

// Shape rule, then balance: a pair CTA carries twice the key tiles of a
// one-tile CTA and the grid has half as many CTAs, so short sequences (few
// query tiles per multiprocessor) leave SMs idle behind the heaviest CTAs.
// The pair schedule is taken when twice the heaviest CTA's key tiles,
// 2 * nq * N, fit into the average key tiles per multiprocessor,
// BH * N^2 * nq (nq + 1) / 2 / num_sms (measured on GB300: at B=1, H=8,
// N=8 the pair forward is 16% slower at S = 8192, where the rule declines
// it, and 4.5% faster at S = 65536).
bool fwd_pair_eligible(const AttnGeom &g, int num_sms) {
    if (!(g.layout == STRIPED_LAYOUT_STRIPED && (g.D == 128 || g.D == 64) && g.seqs.n == 0 && g.N % 2 == 0 &&
          g.L > 0 &&
          g.L % PB == 0) ||
        num_sms < 1)
        return false;
    const double nq = (double)(g.L / PB);
    const double total = (double)g.BH * g.N * g.N * nq * (nq + 1.0) / 2.0;
    const double heaviest = 2.0 * nq * g.N;
    return 2.0 * heaviest * num_sms <= total;
}

template <int HD>
static int launch_pair_hd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const PairParams &p,
                          int64_t nblocks, cudaStream_t stream) {
    static PerDeviceOnce attr_once;
    const int attr = attr_once.get([] {
        return cuda_status(cudaFuncSetAttribute(tc_fwd_pair_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)PairCfg<HD>::kPSmemBytes));
    });
    if (attr != STRIPED_OK) return attr;
    tc_fwd_pair_kernel<HD><<<(unsigned)nblocks, kPThreads, PairCfg<HD>::kPSmemBytes, stream>>>(mq, mk, mv, p);
    return cuda_status(cudaGetLastError());
}

int launch_tc_fwd_pair(const void *q, const void *k, const void *v, void *o, float *lse, const AttnGeom &g,
                       int64_t *tile_stats, cudaStream_t stream) {
    if (!fwd_pair_eligible(g, device_sm_count())) return STRIPED_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv;
    const int64_t bh_kv = g.BH / g.G;
    int st;
    if ((st = make_bf16_map(&mq, q, g.D, g.L, g.N, g.BH, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mk, k, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)) ||
        (st = make_bf16_map(&mv, v, g.D, g.L, g.N, bh_kv, g.stripe_stride, g.stride_bh, 128)))
        return st;
    PairParams p{};
    p.g = g;
    p.o = reinterpret_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.tile_stats = tile_stats;
    p.wc = device_wait_ctl();
    const int64_t nblocks = (g.L / PB) * (g.N / 2) * g.BH;
    if (nblocks > 0x7fffffffll) return STRIPED_ERR_UNSUPPORTED;
    return g.D == 128 ? launch_pair_hd<128>(mq, mk, mv, p, nblocks, stream)
                      : launch_pair_hd<64>(mq, mk, mv, p, nblocks, stream);
}

}  // namespace striped
