// kda_internal.h -- declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Bits of the per-device error word (see kda_check_status).
enum : unsigned { kErrBadSeqlens = 1u, kErrTimeout = 2u };

// Arguments of one prefill or decode launch, already validated on the host.
struct RunParams {
    const void *q, *k, *v, *g, *beta;
    const int32_t *cu_seqlens;  // nullptr: n_seqs sequences of T rows each
    const float *init;          // nullptr: zero initial state
    float *fin;                 // nullptr: final state not stored
    void *o;
    int T;                      // rows per sequence (cu_seqlens == nullptr) or packed rows
    int H;
    int n_seqs;
    unsigned *err;              // device error word
    float gate_bound;           // 0: g holds log-decays; > 0: g holds logits x, g = -gate_bound * sigmoid(x)
};

// Device error word of the current device (created on first use).
unsigned *device_error_word();

// CUDA-core recurrence (decode, fp32 prefill, head sizes without a tensor-core kernel).
cudaError_t launch_recurrent(kda_dtype dtype, int dk, int dv, const RunParams &p, cudaStream_t s);

// Tensor-core chunked prefill (bf16, dk == dv == 128).
bool tc_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p);
cudaError_t launch_tc_prefill(const RunParams &p, cudaStream_t s);

}  // namespace kda
