/*
 * striped.h -- C ABI of libstriped: striped causal attention on one GB300.
 *
 * The method (pages on "Striped Attention: Faster Ring Attention for Causal
 * Transformers"; research.elamur.ai summary page, §Summary and §Key points;
 * pith.science paper page, abstract):
 *   Ring Attention splits a causal sequence of S tokens over N devices in a
 *   ring; key/value blocks circulate so that in round r (0 <= r < N) device d
 *   attends to the key/value stripe of device e = (d - r) mod N.  With a
 *   contiguous split the causal mask leaves some devices fully masked and
 *   others fully kept in each round.  Striped Attention gives device d every
 *   N-th token (positions p with p mod N == d), so each device keeps about
 *   half of every round's work; the output is unchanged because attention is
 *   permutation-equivariant and the permutation is applied once.
 *
 * This library runs the N virtual devices of that ring on ONE GPU: the
 * stripes are slices of one tensor, a "send to the next device" is a pointer
 * to the next stripe, and no collective is issued.
 *
 * Conventions shared by every entry point below:
 *  - Tensors are caller-owned DEVICE pointers, [B, H, S, D] row-major with D
 *    contiguous (16-byte aligned base).  Row order is given by `layout`:
 *      STRIPED_LAYOUT_STRIPED:    row d*L + i holds position i*N + d
 *      STRIPED_LAYOUT_CONTIGUOUS: row r holds position r (device d owns rows
 *                                 [d*L, (d+1)*L))
 *      STRIPED_LAYOUT_ZIGZAG:     row d*L + i holds d*C + i for i < C and
 *                                 (2N-1-d)*C + (i - C) for i >= C, C = S/(2N):
 *                                 device d owns chunk d and chunk 2N-1-d of
 *                                 2N equal chunks (not on the pages; the
 *                                 usual load-balanced placement, kept for
 *                                 comparison).  Attention calls need C to be
 *                                 a multiple of the kernel tile
 *                                 (striped_kernel_tile), else
 *                                 STRIPED_ERR_UNSUPPORTED.
 *    with L = S / N.  LSE arrays are fp32 [B, H, S] in the same row order.
 *  - dtype: STRIPED_BF16 (bf16 storage, fp32 accumulation, tensor cores) or
 *    STRIPED_FP32 (fp32 storage and arithmetic on the CUDA cores).
 *  - Every call is asynchronous on the caller's stream (a cudaStream_t passed
 *    as void*; NULL is the legacy default stream) and allocates nothing.
 *  - Every call returns an int status (STRIPED_OK or a negative code) and
 *    never throws.  Launch failures return STRIPED_ERR_CUDA (the CUDA error
 *    code is kept in striped_last_cuda_error()).  A device-side bounded wait
 *    that expires (2 s by default) records STRIPED_ERR_TIMEOUT in a device
 *    error word that striped_check_error() reads back.  There is ONE error
 *    word per device, shared by every stream and every caller on it: a
 *    timeout is reported to whichever caller next calls
 *    striped_check_error() on that device.
 *  - The library caches per-device addresses (its status block, the
 *    no-allocation scratch array) and kernel attributes the first time it
 *    runs on a device; after cudaDeviceReset() on a device, do not use the
 *    library on that device again in the same process.
 *  - `scale` multiplies the scores q.k (pass 1/sqrt(D) for the usual scaled
 *    dot product).
 *  - `tile_stats`, when not NULL, is an int64 [2][N][N] DEVICE array that
 *    the kernels ADD their processed-tile counts to: [0][r][d] full tiles
 *    and [1][r][d] partial (diagonal) tiles of round r on device d, summed
 *    over all B*H heads.  Tiles are T x T with T from striped_kernel_tile();
 *    fully masked tiles are skipped and not counted.
 */
#ifndef STRIPED_H
#define STRIPED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define STRIPED_OK 0
#define STRIPED_ERR_INVALID_ARG (-1) /* NULL pointer, S % N != 0, N < 1, sizes < 1, bad enum */
#define STRIPED_ERR_UNSUPPORTED (-2) /* head dim / dtype combination not built */
#define STRIPED_ERR_ALIGN (-3)       /* pointer or stride not 16-byte aligned */
#define STRIPED_ERR_CUDA (-4)        /* a CUDA call failed; see striped_last_cuda_error() */
#define STRIPED_ERR_TIMEOUT (-5)     /* a device-side bounded wait expired */
#define STRIPED_ERR_WORKSPACE (-6)   /* workspace NULL or smaller than striped_workspace_size() */

/* dtypes */
#define STRIPED_BF16 0
#define STRIPED_FP32 1

/* row orders */
#define STRIPED_LAYOUT_STRIPED 0
#define STRIPED_LAYOUT_CONTIGUOUS 1
#define STRIPED_LAYOUT_ZIGZAG 2

/*
 * Stripe permutation (§Summary "every N-th token"; §Key points: applied once
 * before the model).  y[b,h,d*L+i,:] = x[b,h,i*N+d,:] for every d < N,
 * i < L.  x and y are [B,H,S,D] device tensors of `dtype`; they must not
 * overlap.  Requires S % N == 0, 16-byte aligned pointers and
 * D * sizeof(dtype) a multiple of 16 bytes (STRIPED_ERR_ALIGN otherwise) of
 * at most 32 KB (STRIPED_ERR_UNSUPPORTED otherwise).  Pure data movement:
 * the result is a bit copy.
 */
int striped_permute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                    int dtype, void *stream);

/* Inverse of striped_permute: y[b,h,i*N+d,:] = x[b,h,d*L+i,:]. */
int striped_unpermute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                      int dtype, void *stream);

/*
 * The same permutation for any `layout`: y[b,h,row,:] = x[b,h,pos(row),:]
 * with pos the layout's row -> position map (see the conventions above;
 * STRIPED_LAYOUT_STRIPED is striped_permute, STRIPED_LAYOUT_CONTIGUOUS a
 * plain copy).  STRIPED_LAYOUT_ZIGZAG requires S % (2N) == 0, else
 * STRIPED_ERR_INVALID_ARG.  Same argument rules and bit-exact result as
 * striped_permute.
 */
int striped_layout_permute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                           int layout, int dtype, void *stream);

/* Inverse of striped_layout_permute: y[b,h,pos(row),:] = x[b,h,row,:]. */
int striped_layout_unpermute(const void *x, void *y, int64_t B, int64_t H, int64_t S, int64_t D,
                             int N, int layout, int dtype, void *stream);

/*
 * Packed variable-length batches (not on the pages; for training on packed
 * documents).  One packed head holds nseq sequences, positions
 * [cu_seqlens[i], cu_seqlens[i+1]) for sequence i; cu_seqlens is a HOST
 * int32 array of nseq + 1 entries with cu_seqlens[0] = 0, S = cu_seqlens[nseq].
 * Each sequence is placed on its own (`layout`, with its own length) and a
 * device's slice of L = S/N rows holds, sequence after sequence, that
 * sequence's L_i = S_i/N rows: row d*L + cu_seqlens[i]/N + j holds position
 * cu_seqlens[i] + pos_i(d*L_i + j).  Tensors are [H, S, D] (one batch
 * entry).  Every S_i must be a positive multiple of N (2N for zig-zag), else
 * STRIPED_ERR_INVALID_ARG; at most 512 sequences (STRIPED_ERR_UNSUPPORTED
 * beyond).  The table is checked on the host and passed to the kernels by
 * value, so nothing is allocated.
 */
int striped_varlen_permute(const void *x, void *y, const int32_t *cu_seqlens, int nseq, int64_t H, int64_t D,
                           int N, int layout, int dtype, void *stream);

/* Inverse of striped_varlen_permute. */
int striped_varlen_unpermute(const void *x, void *y, const int32_t *cu_seqlens, int nseq, int64_t H, int64_t D,
                             int N, int layout, int dtype, void *stream);

/*
 * Causal attention forward over all N ring rounds in one launch (§Summary:
 * each device attends to every circulating key/value stripe; exact result,
 * pith.science abstract).  For each query row of stripe d, rounds
 * r = 0..N-1 visit key stripe e = (d - r) mod N; a (query local i, key local
 * j) pair is kept iff the key's position <= the query's position, which in
 * the striped layout is  j < i  or  (j == i and e <= d),  in the
 * contiguous layout is  e < d,  or  e == d and j <= i,  and in the zig-zag
 * layout follows the chunk positions above.  Fully masked tiles
 * are skipped; partial results of all rounds are merged by the online
 * softmax, so o = softmax(scale * q k^T + causal mask) v exactly up to
 * rounding, and lse = natural-log log-sum-exp of each row's kept scores.
 *  q, k, v: [B,H,S,D] `dtype` inputs in `layout` order.
 *  o:       [B,H,S,D] `dtype` output.      lse: [B,H,S] fp32 output.
 * bf16 requires D == 64 or D == 128; fp32 requires D % 8 == 0 and D <= 128.
 */
int striped_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, int N, int layout, int dtype, float scale,
                     int64_t *tile_stats, void *stream);

/*
 * Grouped-query attention form of striped_attn_fwd (not on the pages; for
 * models whose H query heads share Hkv key/value heads).  q, o: [B,H,S,D];
 * k, v: [B,Hkv,S,D]; lse: [B,H,S].  Query head h of batch entry b attends
 * with key/value head h / (H/Hkv) of the same entry (consecutive query heads
 * share one).  Requires 1 <= Hkv, H % Hkv == 0 (else STRIPED_ERR_INVALID_ARG).
 * Everything else as striped_attn_fwd, which is this call with Hkv = H.
 * tile_stats counts per query head (sums over all B*H).
 */
int striped_attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                         int64_t H, int64_t Hkv, int64_t S, int64_t D, int N, int layout, int dtype,
                         float scale, int64_t *tile_stats, void *stream);

/*
 * Packed variable-length form of striped_attn_fwd_gqa: q, o [H,S,D], k, v
 * [Hkv,S,D], lse [H,S], rows placed as striped_varlen_permute describes.
 * Each sequence attends only within itself (causal inside the sequence):
 * every kernel works on the tiles of one sequence at a time, so tiles across
 * sequences are neither computed nor counted.  Every S_i must also be a
 * whole number of kernel tiles per device: S_i a multiple of N*T (2N*T for
 * zig-zag), T from striped_kernel_tile(), else STRIPED_ERR_UNSUPPORTED.
 */
int striped_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int32_t *cu_seqlens, int nseq, int64_t H, int64_t Hkv, int64_t D, int N,
                            int layout, int dtype, float scale, int64_t *tile_stats, void *stream);

/* Bytes of device workspace striped_attn_bwd needs for these sizes (fp32 dQ
 * accumulator and per-row softmax statistics padded to whole tiles), or 0
 * for invalid sizes. */
size_t striped_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D, int N, int dtype);

/*
 * Backward of striped_attn_fwd (training use, §Summary).  Given the forward
 * inputs, its outputs o and lse, and the output cotangent dO, writes
 *   dq = scale * dS k,  dk = scale * dS^T q,  dv = P^T dO,
 * with P = exp(scale q k^T - lse) on kept pairs, dS = P * (dO v^T - Delta)
 * and Delta_p = <dO_p, o_p>.  Same tile skipping as the forward.
 *  q,k,v,o,dO: [B,H,S,D] `dtype`;  lse: [B,H,S] fp32 from the forward.
 *  dq,dk,dv:   [B,H,S,D] `dtype` outputs (fully overwritten).
 *  workspace:  caller-owned device buffer of >= striped_workspace_size()
 *              bytes, 256-byte aligned; its contents on entry are ignored.
 */
int striped_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dO, void *dq, void *dk, void *dv, void *workspace,
                     size_t ws_bytes, int64_t B, int64_t H, int64_t S, int64_t D, int N,
                     int layout, int dtype, float scale, int64_t *tile_stats, void *stream);

/*
 * Backward of striped_attn_fwd_gqa.  q, o, dO, dq: [B,H,S,D]; k, v, dk, dv:
 * [B,Hkv,S,D].  dk and dv of a key/value head are the sums over the H/Hkv
 * query heads that read it (accumulated on chip, no atomics); the workspace
 * is striped_workspace_size(B, H, S, D, N, dtype) (dQ is per query head).
 * striped_attn_bwd is this call with Hkv = H.
 */
int striped_attn_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dO, void *dq, void *dk, void *dv, void *workspace,
                         size_t ws_bytes, int64_t B, int64_t H, int64_t Hkv, int64_t S, int64_t D, int N,
                         int layout, int dtype, float scale, int64_t *tile_stats, void *stream);

/*
 * Backward of striped_attn_fwd_varlen (same packed layout and limits); the
 * workspace is striped_workspace_size(1, H, S, D, N, dtype).
 */
int striped_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                            const void *dO, void *dq, void *dk, void *dv, void *workspace, size_t ws_bytes,
                            const int32_t *cu_seqlens, int nseq, int64_t H, int64_t Hkv, int64_t D, int N,
                            int layout, int dtype, float scale, int64_t *tile_stats, void *stream);

/*
 * striped_attn_bwd for callers that cannot allocate device memory (the paper
 * has no counterpart; this is a library convenience).  Same arguments,
 * results and tile counters as striped_attn_bwd, minus the workspace: the
 * scratch lives in a fixed 48 MiB device array inside the library, present
 * on every GPU that loads it until the process exits.  For callers whose
 * device memory is owned by an allocator or budget they cannot extend, or
 * who must keep cudaMalloc off their hot path.
 *  - Returns STRIPED_ERR_WORKSPACE when striped_workspace_size(B,H,S,D,N,dtype)
 *    exceeds 48 MiB (bf16, D = 128: B*H*S up to about 96,000 rows).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on one device share the array: calls that overlap on the GPU
 *    race and give wrong results.  Nothing needs clearing by the caller.
 */
int striped_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dO, void *dq, void *dk, void *dv,
                             int64_t B, int64_t H, int64_t S, int64_t D, int N, int layout,
                             int dtype, float scale, int64_t *tile_stats, void *stream);

/*
 * One ring round of one virtual device (§Summary: per round, a device's
 * query block attends to the key/value block it currently holds; the
 * partial results are merged into running output statistics).
 * Computes the partial result (O_r, LSE_r) of query stripe d against key
 * stripe e under the mask of `layout` (see striped_attn_fwd), then merges it
 * into the running accumulator with the log-sum-exp rule
 *     lse' = log(exp(lse_acc) + exp(LSE_r)),
 *     o'   = exp(lse_acc - lse') o_acc + exp(LSE_r - lse') O_r;
 * a side whose LSE is -inf (no kept key yet) contributes nothing.  With
 * first_round != 0 the accumulator is overwritten by (O_r, LSE_r).
 *  q_d, k_e, v_e: stripe slices, L rows per (b,h), consecutive (b,h) slices
 *                 `stride_bh` ELEMENTS apart (S*D for slices of a full
 *                 [B,H,S,D] tensor); `dtype`.
 *  o_acc:   fp32, same geometry and stride as q_d (running normalised O).
 *  lse_acc: fp32, L per (b,h), `lse_stride_bh` elements apart (natural log).
 *  o_out:   optional (NULL to skip) `dtype` copy of the merged O, same
 *           geometry as q_d.
 *  tile_stats gets this round's counts at [.][r][d] with r = (d - e) mod N.
 */
int ring_round_fwd(const void *q_d, const void *k_e, const void *v_e, float *o_acc, float *lse_acc,
                   void *o_out, int d, int e, int64_t B, int64_t H, int64_t L, int64_t D, int N,
                   int64_t stride_bh, int64_t lse_stride_bh, int layout, int dtype, float scale,
                   int first_round, int64_t *tile_stats, void *stream);

/*
 * The backward of one ring round, for a ring of N processes that each hold
 * one stripe (§Summary: key/value blocks circulate around the ring; here
 * the gradients of a key/value block travel with it and are summed by every
 * device it visits, then return to its owner).  bf16 only
 * (STRIPED_ERR_UNSUPPORTED for fp32).  Every block is the device's own
 * CONTIGUOUS [B, H, L, D] tensor (L = S/N rows of one stripe, in the
 * layout's row order; 16-byte aligned), lse_d fp32 [B, H, L].
 *
 * ring_bwd_workspace_size: bytes of the per-device statistics workspace
 * (softmax statistics of the device's L query rows padded to 128-row tiles),
 * or 0 for invalid sizes.
 *
 * ring_bwd_prepare: once per backward, on device d: writes the statistics
 * of its query block (LSE and Delta = <dO, O> per row) into `workspace` and
 * zeroes its fp32 dQ sum dq_acc_d [B, H, L, D].
 *
 * ring_round_bwd: device d's round against the key/value block of stripe e
 * (the block it holds in ring round (d - e) mod N): adds the round's dQ
 * share into dq_acc_d and the round's dK, dV shares (scale applied to dK)
 * into the fp32 sums dk_acc_e, dv_acc_e [B, H, L, D] that travel with the
 * block; with first_round != 0 the sums are overwritten instead (the
 * block's first round, on its own device).  Same mask and tile skipping as
 * striped_attn_bwd; tile_stats gets the round's counts at [.][r][d].
 *
 * ring_bwd_finish: out = bf16(mul * acc) for n fp32 values (n a multiple of
 * 8): dQ with mul = scale, the returned dK and dV sums with mul = 1.
 */
size_t ring_bwd_workspace_size(int64_t B, int64_t H, int64_t L, int64_t D, int dtype);
int ring_bwd_prepare(const void *o_d, const float *lse_d, const void *dO_d, void *workspace, size_t ws_bytes,
                     float *dq_acc_d, int64_t B, int64_t H, int64_t L, int64_t D, int dtype, void *stream);
int ring_round_bwd(const void *q_d, const void *k_e, const void *v_e, const void *dO_d, const void *workspace,
                   size_t ws_bytes, float *dq_acc_d, float *dk_acc_e, float *dv_acc_e, int d, int e, int64_t B,
                   int64_t H, int64_t L, int64_t D, int N, int layout, int dtype, float scale, int first_round,
                   int64_t *tile_stats, void *stream);
int ring_bwd_finish(const float *acc, void *out, int64_t n, int dtype, float mul, void *stream);

/* Tile edge T (queries x keys) the kernels for (dtype, D) skip and count
 * with; writes *Tq and *Tk.  Returns STRIPED_ERR_UNSUPPORTED if no kernel. */
int striped_kernel_tile(int dtype, int64_t D, int *Tq, int *Tk);

/* Host-only: how many query tiles one CTA of striped_attn_fwd /
 * striped_attn_fwd_gqa runs for this problem on a GPU with `num_sms`
 * multiprocessors: 2 when the stripes d and d + 1 share one K/V stream (bf16,
 * D = 64 or 128, striped placement, L = S/N a whole number of 128-row tiles,
 * N even) and the grid stays balanced -- twice the heaviest CTA's key tiles,
 * 2 * (L/128) * N, at most the average key tiles per multiprocessor -- else
 * 1.  Both schedules do the same arithmetic in the same order (measured
 * bit-identical at D = 128).  Returns 1 or 2,
 * or STRIPED_ERR_INVALID_ARG / STRIPED_ERR_UNSUPPORTED for arguments the
 * forward rejects (num_sms < 1 is invalid). */
int striped_fwd_query_tiles_per_cta(int64_t B, int64_t H, int64_t S, int64_t D, int N, int layout, int dtype,
                                    int num_sms);

/*
 * Host-only, exact: per-(b,h) processed-tile table of the ring (§Summary
 * and §Key points "Imbalance": per-round work per device).  full and
 * partial are HOST int64 arrays [N rounds][N devices]; a Tq x Tk tile of
 * round r on device d (keys of stripe e = (d - r) mod N) is "full" when all
 * of its in-range pairs are kept, "partial" when some are, and not counted
 * when none are.  Either output may be NULL.
 */
int striped_tile_counts(int64_t S, int N, int Tq, int Tk, int layout, int64_t *full,
                        int64_t *partial);

/* Host-only: modelled ring critical path = sum over rounds of the largest
 * per-device tile count (each round runs at the pace of its slowest
 * device, §Summary).  Returns < 0 (a status code) on invalid arguments. */
int64_t striped_critical_path(int64_t S, int N, int Tq, int Tk, int layout);

/* Host-only: striped_tile_counts for a packed batch (cu_seqlens a HOST
 * int32 array of nseq + 1 entries, as for striped_attn_fwd_varlen): each
 * sequence is placed and tiled on its own, so the table is the sum of the
 * sequences' tables; per packed head. */
int striped_tile_counts_varlen(const int32_t *cu_seqlens, int nseq, int N, int Tq, int Tk, int layout,
                               int64_t *full, int64_t *partial);

/* Host-only: modelled ring critical path of a packed batch (each round runs
 * at the pace of the device with the most tiles over all its sequences). */
int64_t striped_critical_path_varlen(const int32_t *cu_seqlens, int nseq, int N, int Tq, int Tk, int layout);

/* Synchronises `stream`, then reads and clears the error word of the
 * current device (one per device, not per stream; see the conventions).
 * Returns STRIPED_OK, STRIPED_ERR_TIMEOUT, STRIPED_ERR_ALIGN or
 * STRIPED_ERR_CUDA. */
int striped_check_error(void *stream);

/* Human-readable name of a status code (static string). */
const char *striped_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by the library. */
int striped_last_cuda_error(void);

/*
 * Self-test of the device-side timeout path: launches one tiny kernel that
 * waits, with a bound of `spins` polls, on a device flag that nothing sets;
 * when the bound runs out it records STRIPED_ERR_TIMEOUT in the device error
 * word and returns.  Read the result with striped_check_error().  No fault,
 * trap or hang is involved.
 */
int striped_selftest_timeout(int64_t spins, void *stream);

/*
 * TEST HOOK (not for production use): checks that the attention kernels'
 * own bounded waits end, report STRIPED_ERR_TIMEOUT and leave the device
 * usable.  Synchronises the current device, then sets for every later launch
 * on it:
 *  - wait_limit_ns: the bound of every device-side wait (<= 0 restores the
 *    default 2 s);
 *  - fault: STRIPED_FAULT_NONE, or STRIPED_FAULT_FWD_SKIP_KV (the forward
 *    kernels' TMA producer never loads its first K/V tile) or
 *    STRIPED_FAULT_BWD_SKIP_Q (the tensor-core backward's producer never
 *    loads its first Q tile).  Every wait on the missing tile runs out; each
 *    CTA then records the timeout, waits (bounded) for its own copies and
 *    tensor-core operations in flight, frees its tensor memory and returns.
 *    No fault, trap or hang is involved; results of such a launch are
 *    garbage.
 * Restore with striped_test_inject(STRIPED_FAULT_NONE, 0).  Returns
 * STRIPED_ERR_INVALID_ARG for an unknown fault, else STRIPED_OK or
 * STRIPED_ERR_CUDA.
 */
#define STRIPED_FAULT_NONE 0
#define STRIPED_FAULT_FWD_SKIP_KV 1
#define STRIPED_FAULT_BWD_SKIP_Q 2
int striped_test_inject(int fault, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* STRIPED_H */
