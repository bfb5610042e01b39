// common.cuh -- device helpers shared by the libstriped kernels (sm_103a).
//
//  * the per-round tile schedule of the ring (which key tiles a query tile
//    visits in round r, and which of them need a mask);
//  * bounded waits that record a timeout in the device status block instead
//    of hanging;
//  * thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the
//    5th-generation tensor core (tcgen05: TMEM alloc, mma, commit, ld, st).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "striped.h"

namespace striped {

// --------------------------------------------------------------------------
// bounded waits; a timeout is recorded in the library's device status block
// (owned by api.cu, passed to every kernel as a pointer)
// --------------------------------------------------------------------------
// The library's device-side status word: the status the next
// striped_check_error() returns (one per device, shared by every stream and
// caller on it).
struct DeviceStatus {
    int error;
};
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
constexpr int kInjectNone = STRIPED_FAULT_NONE;
constexpr int kInjectFwdSkipKV = STRIPED_FAULT_FWD_SKIP_KV;  // forward TMA producers skip their first K/V tile
constexpr int kInjectBwdSkipQ = STRIPED_FAULT_BWD_SKIP_Q;    // backward TMA producers skip their first Q tile

// What every wait of a launch needs, passed by value in the kernel
// parameters (so a wait reads nothing from memory): where to record a
// failure, the bound of every mbarrier wait (wall-clock time read from
// %globaltimer; every legitimate wait is microseconds) and the test hook
// that makes one kind of kernel skip one of its own loads (kInject*, 0
// outside tests).
struct WaitCtl {
    DeviceStatus *st;
    unsigned long long limit_ns;
    int inject;
};

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(DeviceStatus *st, int code) {
    if (st) atomicExch(&st->error, code);
}

__device__ __forceinline__ void record_timeout(const WaitCtl &w) { record_error(w.st, STRIPED_ERR_TIMEOUT); }

// --------------------------------------------------------------------------
// tile schedule
// --------------------------------------------------------------------------
// For a query tile (stripe d, tile a) and a key stripe e, the key tiles
// b = 0 .. nfull-1 are kept in full; if has_diag, tile b = nfull is partially
// kept with the mask  key_col <= query_row + diag_off  (local columns and
// rows inside the tile).  Positions: striped row d*L+i holds i*N+d, so the
// pair (i, j) is kept iff j*N+e <= i*N+d, i.e. j <= i - 1 + [e <= d];
// contiguous rows hold their own position, so the pair is kept iff e < d, or
// e == d and j <= i.  Zig-zag rows i < C hold d*C + i and rows i >= C hold
// (2N-1-d)*C + i - C (C = L/2, a multiple of T, so with c = nk/2 tiles per
// chunk, tiles a < c lie in chunk d and tiles a >= c in chunk 2N-1-d); a
// query chunk keeps every key chunk of lower index in full and the causal
// triangle of its own.  `rows_a` is the number of in-range rows of tile a
// (T, or fewer for the last, ragged tile); key tiles have the same edge T.
struct RoundSpan {
    int nfull;     // fully kept key tiles b = 0 .. nfull-1
    int has_diag;  // 1 if tile b = nfull is partially kept
    int diag_off;  // keep iff key_col <= query_row + diag_off  (-1 or 0)
};

__host__ __device__ __forceinline__ RoundSpan round_span(int layout, int d, int e, int a, int nk,
                                                         int rows_a) {
    RoundSpan s{0, 0, 0};
    if (layout == STRIPED_LAYOUT_ZIGZAG) {
        const int c = nk / 2;
        if (e == d) {  // own chunks: everything below the diagonal tile a
            s.nfull = a;
            s.has_diag = 1;
        } else if (a < c) {  // query chunk d: key chunk e < d only
            s.nfull = (e < d) ? c : 0;
        } else {  // query chunk 2N-1-d: key chunk e always, 2N-1-e if e > d
            s.nfull = (e > d) ? 2 * c : c;
        }
        return s;
    }
    if (layout == STRIPED_LAYOUT_STRIPED) {
        const int off = (e <= d) ? 0 : -1;
        s.nfull = a;
        if (rows_a >= 2) {
            s.has_diag = 1;
            s.diag_off = off;
        } else if (off == 0) {
            s.nfull = a + 1;  // a 1x1 diagonal tile holding a kept pair
        }
    } else {
        if (e < d) {
            s.nfull = nk;
        } else if (e == d) {
            s.nfull = a;
            if (rows_a >= 2) {
                s.has_diag = 1;
                s.diag_off = 0;
            } else {
                s.nfull = a + 1;
            }
        }
    }
    return s;
}

// Transposed view for the backward pass: for key tile (stripe e, tile b) and
// query stripe d, the query tiles that see it are a in [a_lo, nq); tile a_lo
// is the partially kept diagonal when has_diag (mask as above), every other
// tile in the range is fully kept.
struct QuerySpan {
    int a_lo;
    int has_diag;
    int diag_off;
};

__host__ __device__ __forceinline__ QuerySpan query_span(int layout, int d, int e, int b, int nq,
                                                         int rows_b) {
    QuerySpan s{nq, 0, 0};
    if (layout == STRIPED_LAYOUT_ZIGZAG) {
        const int c = nq / 2;
        if (e == d) {  // own chunks: the diagonal tile b and every tile after it
            s.a_lo = b;
            s.has_diag = 1;
        } else if (b < c) {  // key chunk e: all of query chunk 2N-1-d, and chunk d if e < d
            s.a_lo = (e < d) ? 0 : c;
        } else {  // key chunk 2N-1-e: only query chunk 2N-1-d, and only if e > d
            s.a_lo = (e > d) ? c : nq;
        }
        return s;
    }
    if (layout == STRIPED_LAYOUT_STRIPED) {
        const int off = (e <= d) ? 0 : -1;
        if (rows_b >= 2) {
            s.a_lo = b;
            s.has_diag = 1;
            s.diag_off = off;
        } else {
            s.a_lo = (off == 0) ? b : b + 1;
        }
    } else {
        if (d > e) {
            s.a_lo = 0;
        } else if (d == e) {
            s.a_lo = b;
            if (rows_b >= 2) {
                s.has_diag = 1;
                s.diag_off = 0;
            }
        }
    }
    if (s.a_lo > nq) s.a_lo = nq;
    return s;
}

// The packed sequence holding tile (or row) x of a device's slice, in units
// of `unit` rows: its first unit and its length in units.  A dense launch
// (table size 0) is one sequence of `total` units.  Binary search over the
// table in the kernel parameters (uniform across the CTA).
struct SeqSpan {
    int start, count;
};

template <typename Table>
__device__ __forceinline__ SeqSpan seq_of(const Table &t, int x, int unit, int total) {
    if (t.n == 0) return SeqSpan{0, total};
    int lo = 0, hi = t.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.row_start[mid] / unit <= x) lo = mid;
        else hi = mid - 1;
    }
    const int s0 = t.row_start[lo] / unit;
    return SeqSpan{s0, t.row_start[lo + 1] / unit - s0};
}

__host__ __device__ __forceinline__ int ring_round_of(int d, int e, int N) {
    return ((d - e) % N + N) % N;
}

// --------------------------------------------------------------------------
// shared-memory address + mbarrier
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false (and the device
// status set to STRIPED_ERR_TIMEOUT) if the bound runs out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &w) {
    for (int it = 0; it < 64; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_timer_ns() - t0 > w.limit_ns) break;
    }
    record_timeout(w);
    return false;
}

// --------------------------------------------------------------------------
// TMA
// --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Plain bulk copy global -> shared of `bytes` (multiple of 16, both
// addresses 16-byte aligned), completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Element-wise add of a shared-memory box into global memory through the
// tensor map (out-of-range rows are skipped), tracked by the bulk group of
// the issuing thread.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2,
                                                  int c3) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%1, %2, %3, %4}], [%5];" ::"l"(reinterpret_cast<uint64_t>(m)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The shared-memory sources of this thread's bulk groups may be reused.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------------------
// tcgen05
// --------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B
// format (1 = bf16), 15 A major (0 = K, 1 = MN), 16 B major, [17,23) N>>3,
// [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   bits [0,14) start address >> 4, [16,30) leading byte offset >> 4,
//   [32,46) stride byte offset >> 4, [46,48) = 1 (descriptor version),
//   [61,64) = 2 (128-byte swizzle).  Operand tiles are 1024-byte aligned.
// K-major operand (rows of 64 bf16 = 128 B, 8-row atoms of 1024 B): SBO is
// the 8-row group stride (1024); LBO is unused.  MN-major operand (128-B
// rows of 64 MN-contiguous elements, one row per K index, 8 K-rows per
// atom): LBO is the stride between 64-element MN blocks, SBO the stride
// between 8-K-row groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane
// (base lane + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Wait for outstanding tcgen05.ld of this thread; the registers are passed
// through so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 lanes x 16 columns (x16 variants of the above).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Wait for outstanding tcgen05.ld, passing two register sets through.
__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&a)[32], uint32_t (&b)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                   "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                   "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]),
                   "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]),
                   "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]),
                   "+r"(a[30]), "+r"(a[31]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]),
                   "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]),
                   "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------------------------
// small numeric helpers
// --------------------------------------------------------------------------
// 2^x with the SFU instruction (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Paired fp32 arithmetic (two lanes in one 64-bit register pair, each lane
// an IEEE fp32 operation rounded to nearest): half the instructions of two
// scalar operations with bit-identical results.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {  // a * b + c
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// max of three fp32 values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_f32(float *addr, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

}  // namespace striped
