// internal.h -- declarations shared between the host entry points (api.cu)
// and the kernel launchers.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "striped.h"

namespace striped {

// Records a failed CUDA call so striped_last_cuda_error() can report it and
// maps it to a status code.
int cuda_status(cudaError_t err);

// A status computed once per device, under a lock: kernel attributes (the
// dynamic shared-memory opt-in) are per device, so a process that launches
// on several GPUs sets them on each.
constexpr int kMaxDevices = 256;
class PerDeviceOnce {
  public:
    template <typename F>
    int get(F &&fn) {
        int dev = 0;
        const cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_status(e);
        if (dev < 0 || dev >= kMaxDevices) return STRIPED_ERR_UNSUPPORTED;
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            status_[dev] = fn();
            done_[dev] = true;
        }
        return status_[dev];
    }

  private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
    int status_[kMaxDevices] = {};
};

// Device address of the library's status word on the current device (where
// bounded waits record STRIPED_ERR_TIMEOUT), or nullptr on failure.  Looked
// up once per device under a lock.
struct DeviceStatus;
DeviceStatus *device_status();

// The wait control of a launch on the current device: its status word, the
// wait bound and the test hook as set by striped_test_inject (defaults: 2 s,
// none).
struct WaitCtl;
WaitCtl device_wait_ctl();

// Geometry of one attention launch.  Every tensor is addressed as
// [BH][N stripes][L rows][D] with stripe e of head bh starting at element
// bh*stride_bh + e*stripe_stride (stripe_stride = L*D for full tensors,
// 0 when the pointers are already the stripe slices of one round).
// Packed variable-length batches: the sequences of one packed head, as the
// first row of each inside every device's slice (row_start[i] =
// cu_seqlens[i] / N, row_start[n] = L).  n = 0 means one sequence per
// (batch, head), the dense case.  Carried by value in the kernel parameters.
constexpr int kMaxSeqs = 512;
struct SeqTable {
    int n;
    int row_start[kMaxSeqs + 1];
};

// Grouped-query attention: query head bh (of B*H) reads key/value head
// bh / G (of B*H/G), i.e. G consecutive query heads share one; G = 1 is
// plain multi-head attention.
struct AttnGeom {
    int64_t BH, L, D;
    int64_t G;                  // query heads per key/value head
    int N;
    int layout;
    int64_t stride_bh;          // elements between heads (q/k/v/o)
    int64_t stripe_stride;      // elements between stripes
    int64_t lse_stride_bh;      // elements between heads of lse
    int64_t lse_stripe_stride;  // elements between stripes of lse
    float scale;
    SeqTable seqs;              // packed sequences (seqs.n == 0: dense)
};

// ---- permute.cu
int launch_stripe_permute(const void *x, void *y, int64_t BH, int64_t S, int64_t row_bytes, int N,
                          int layout, bool gather, const SeqTable &seqs, cudaStream_t stream);

// ---- attn_simt.cu (fp32 CUDA-core path, tile edge kSimtTile)
constexpr int kSimtTile = 16;
int launch_simt_fwd(const float *q, const float *k, const float *v, float *o, float *lse,
                    const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream);
int launch_simt_round(const float *q_d, const float *k_e, const float *v_e, float *o_acc,
                      float *lse_acc, float *o_out, int d, int e, int first, const AttnGeom &g,
                      int64_t *tile_stats, cudaStream_t stream);
int launch_simt_bwd(const float *q, const float *k, const float *v, const float *o,
                    const float *lse, const float *dO, float *dq, float *dk, float *dv,
                    float *delta_ws, const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream);

// ---- attn_fwd_tc.cu / attn_bwd_tc.cu (bf16 tensor-core path, tile 128)
constexpr int kTcTile = 128;
int launch_tc_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                  const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream);
// attn_fwd_pair.cu: the batched forward with two query tiles (stripes d and
// d+1) per CTA; STRIPED_ERR_UNSUPPORTED unless fwd_pair_eligible(g, sms)
// with the current device's multiprocessor count.
bool fwd_pair_eligible(const AttnGeom &g, int num_sms);
// Multiprocessor count of the current device (queried once per device; 152
// if the query fails).
int device_sm_count();
int launch_tc_fwd_pair(const void *q, const void *k, const void *v, void *o, float *lse,
                       const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream);
int launch_tc_round(const void *q_d, const void *k_e, const void *v_e, float *o_acc, float *lse_acc,
                    void *o_out, int d, int e, int first, const AttnGeom &g, int64_t *tile_stats,
                    cudaStream_t stream);
int launch_tc_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dO, void *dq, void *dk, void *dv, float *dq_acc, float *stats,
                  const AttnGeom &g, int64_t *tile_stats, cudaStream_t stream);

// One ring round of the backward (every block its own contiguous
// [BH][L][D] tensor): the statistics of device d's query block and its
// zeroed fp32 dQ sum; the round itself (dQ added into dq_acc, dK and dV
// added into -- or with first, written to -- the fp32 sums of key block
// e); and the final out = bf16(mul * sum) of n8 * 8 values.
int launch_round_bwd_prepare(const void *o_d, const float *lse_d, const void *dO_d, float *stats, float *dq_acc,
                             const AttnGeom &g, cudaStream_t stream);
int launch_tc_round_bwd(const void *q_d, const void *k_e, const void *v_e, const void *dO_d, const float *stats,
                        float *dq_acc, float *dk_acc, float *dv_acc, int d, int e, int first, const AttnGeom &g,
                        int64_t *tile_stats, cudaStream_t stream);
int launch_scale_to_bf16(const float *acc, void *out, int64_t n8, float mul, cudaStream_t stream);

// bf16 tensor viewed as [BH][N][L][D] -> 4-D tensor map with boxes of
// 64 elements x box_rows rows, 128-byte swizzle, zero fill out of range.
// Returns a status code.
int make_bf16_map(CUtensorMap *map, const void *base, int64_t D, int64_t L, int64_t N, int64_t BH,
                  int64_t stripe_stride, int64_t stride_bh, int box_rows);
// Same for fp32 tensors: boxes of 32 elements (128 bytes) x box_rows rows.
int make_f32_map(CUtensorMap *map, const void *base, int64_t D, int64_t L, int64_t N, int64_t BH,
                 int64_t stripe_stride, int64_t stride_bh, int box_rows);

}  // namespace striped
