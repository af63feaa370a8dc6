// kda_internal.h -- declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Bits of the per-device error word (see kda_check_status).
enum : unsigned { kErrBadSeqlens = 1u, kErrTimeout = 2u, kErrBadIndex = 4u };

// Arguments of one prefill or decode launch, already validated on the host.
struct RunParams {
    const void *q, *k, *v, *g, *beta;
    const int32_t *cu_seqlens;  // nullptr: n_seqs sequences of T rows each
    const float *init;          // nullptr: zero initial state
    float *fin;                 // nullptr: final state not stored
    void *o;
    int T;                      // rows per sequence (cu_seqlens == nullptr) or packed rows
    int H;
    int dk;                     // head size of the tensors (dk == dv); the tensor-core kernel pads it to 128
    int n_seqs;
    unsigned *err;              // device error word
    float gate_bound;           // 0: g holds log-decays; > 0: g holds logits x, g = -gate_bound * sigmoid(x)
    // Tensor-core kernel only (segment transitions of the segmented long-sequence prefill):
    bool zero_v;                // v taken as 0 (the v tensor is not read)
    bool identity_init;         // initial state = identity (needs d_k == d_v; init is not read)
    // Options of both the tensor-core and the recurrent kernel:
    bool qk_l2norm;             // q and k rows divided by sqrt(sum x^2 + 1e-6) in the kernel
    const int32_t *init_idx;    // non-null: init is a pool; sequence n starts from state init_idx[n] (< 0: zero)
    const int32_t *fin_idx;     // non-null: fin is a pool; sequence n ends in state fin_idx[n] (< 0: not written)
    int pool;                   // states in the pool(s) when an index array is given
    const void *out_gate;       // non-null: o is multiplied by sigmoid(out_gate) (same layout and dtype as o)
    // Tensor-core kernel only (launch order of packed sequences; passes of the split prefill):
    const int32_t *order;       // non-null: CTA block b / H runs sequence order[b / H] (a permutation)
    int max_chunks;             // > 0: only the first max_chunks chunks of every sequence are run
    const uint8_t *skip;        // non-null: the CTA of (sequence n, head h) exits at once if skip[n*H + h]
    // Diagnostic (kda_prefill_debug_dump): the chunkwise intermediates of the first (sequence, head).
    float *dump;                // non-null: plain bf16 d = 128 only
    int dump_chunks;
};

// Device error word of the current device (created on first use).
unsigned *device_error_word();

// CUDA-core recurrence (decode, fp32 prefill, head sizes without a tensor-core kernel).
cudaError_t launch_recurrent(kda_dtype dtype, int dk, int dv, const RunParams &p, cudaStream_t s);

// Tensor-core chunked prefill (bf16, dk == dv == 128).
bool tc_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p);
cudaError_t launch_tc_prefill(const RunParams &p, cudaStream_t s);

// Tensor-core chunked prefill in tf32 (fp32, dk == dv in {32, 64}, without the L2 normalisation
// and the output gate).
bool tf32_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p);
cudaError_t launch_tf32_prefill(const RunParams &p, cudaStream_t s);

// TMA map of a bf16 [rows, H, d] tensor in boxes of 64 rows x 64 channels (128-byte swizzle), the
// tile of the tensor-core kernels (channels past d read as zeros and are not written). False if the
// driver's encoder is unavailable or rejects it.
bool encode_row_tile_map(CUtensorMap *map, const void *base, long long rows, int H, int d = 128);

// Segmented prefill of few long sequences (see kda_segmented.cu): workspace bytes it needs for
// this call (0: the call is not eligible), and the launch sequence.
size_t segmented_workspace_bytes(kda_dtype dtype, int B, int T, int H, int dk, int dv, bool varlen);
// The same plan for a GPU with `sms` SMs (host arithmetic only): segments per sequence (0: not
// split), rows per segment and workspace bytes.
void segmented_plan_for(int B, int T, int H, int sms, int *P, int *Ls, size_t *bytes);
cudaError_t launch_segmented_prefill(const RunParams &p, int B, void *workspace, size_t workspace_bytes,
                                     cudaStream_t s);
// The same for packed sequences (cu_seqlens): the segments are planned on the device from the lengths.
// Workspace bytes on a GPU with `sms` SMs (0: such a call is not split), and the launch sequence.
size_t segmented_packed_workspace_bytes_for(kda_dtype dtype, int n_seqs, int T, int H, int dk, int dv, int sms);
cudaError_t launch_segmented_packed_prefill(const RunParams &p, void *workspace, size_t workspace_bytes,
                                            cudaStream_t s);

// Longest-first launch order of packed sequences (see kda_api.cu): workspace bytes and the sort.
constexpr int kMaxOrderedSeqs = 4096;
size_t order_workspace_bytes(kda_dtype dtype, int dk, int dv, int n_seqs);
cudaError_t launch_order_by_length(const int32_t *cu_seqlens, int n_seqs, int32_t *order, cudaStream_t s);

// Backward pass (see kda_backward.cu): workspace bytes for the state checkpoints, and the launch.
size_t backward_workspace_bytes(int T_total, int n_seqs, int H, int d);
size_t backward_chunked_workspace_bytes(int T_total, int n_seqs, int H);
cudaError_t launch_backward_chunked(kda_dtype dtype, const RunParams &p, const void *d_o, const float *d_fin,
                                    float *dq, float *dk, float *dv, float *dg, float *dbeta, float *d_init,
                                    void *ws, cudaStream_t s);
cudaError_t launch_backward(kda_dtype dtype, int d, const RunParams &p, const void *d_o, const float *d_fin,
                            float *dq, float *dk, float *dv, float *dg, float *dbeta, float *d_init, void *ws,
                            cudaStream_t s);

// Element offset of the state of (sequence n, head h) in a state tensor of d x d blocks, or -1
// when the sequence has none there. Without an index array the tensor holds one state per
// sequence; with one it is a pool of `pool` states and idx[n] picks the slot (negative: none; at
// or past the pool end: none, and kErrBadIndex is raised).
__device__ __forceinline__ long long state_slot_offset(const int32_t *idx, int pool, int n, int H, int h,
                                                       int d, unsigned *err) {
    long long slot = n;
    if (idx) {
        slot = idx[n];
        if (slot < 0) return -1;
        if (slot >= pool) {
            atomicOr(err, kErrBadIndex);
            return -1;
        }
    }
    return (slot * H + h) * (long long)d * d;
}

}  // namespace kda
