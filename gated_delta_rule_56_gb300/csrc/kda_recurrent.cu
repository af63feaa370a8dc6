// kda_recurrent.cu -- the KDA recurrence token by token on CUDA cores.
//
// Serves the single-token decode step (HBM-bound: each head's fp32 state is streamed
// through registers once), the fp32 prefill, and any head size the tensor-core chunked
// kernel does not take. Per (sequence, head) and token, following "Kimi Delta Attention:
// the linear core" (maidul-haque blog) -- decay each key channel, remove the value the key
// currently reads, write the corrected value, read out with the query:
//     S' = Diag(exp g) S;  u = beta (v - S'^T k);  S = S' + k u^T;  o = S^T q = S'^T q + (q.k) u
//
// Work split: one CTA of 8 warps per (sequence, head). Warp w owns key rows
// [w*DK/8, (w+1)*DK/8) of the state, lane l owns value columns [l*DV/32, (l+1)*DV/32), so
// a warp reads whole 512-byte state rows with 16-byte vector loads (coalesced) and the
// column reductions over key rows are an in-register sum plus one cross-warp pass through
// shared memory. State loads and stores use the streaming cache hint: each element is read
// once and written once.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float load_elem(const float *p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <int CPL>
__device__ __forceinline__ void load_state(const float *p, float (&out)[CPL]) {
    if constexpr (CPL == 4) {
        const float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
        out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
    } else if constexpr (CPL == 2) {
        const float2 x = __ldcs(reinterpret_cast<const float2 *>(p));
        out[0] = x.x; out[1] = x.y;
    } else {
        out[0] = __ldcs(p);
    }
}

template <int CPL>
__device__ __forceinline__ void store_state(float *p, const float (&x)[CPL]) {
    if constexpr (CPL == 4) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    } else if constexpr (CPL == 2) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(x[0], x[1]));
    } else {
        __stcs(p, x[0]);
    }
}

// EXT: the instance that also serves q/k L2 normalisation and the output gate; the plain
// instance carries neither (the decode step runs at the register limit).
template <typename Tin, int DK, int DV, bool EXT>
__global__ void __launch_bounds__(kThreads, 2) recurrent_kernel(RunParams p) {
    static_assert(DK % kWarps == 0 && DV % 32 == 0 && DK + DV <= kThreads, "head size");
    constexpr int RPW = DK / kWarps;  // key rows per warp
    constexpr int CPL = DV / 32;      // value columns per lane
    const int H = p.H;
    const int h = blockIdx.x % H;
    const int n = blockIdx.x / H;
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;

    long long bos, eos;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > p.T || (n == 0 && bos != 0) ||
            (n == p.n_seqs - 1 && eos != p.T)) {
            if (tid == 0) atomicOr(p.err, kErrBadSeqlens);
            return;
        }
    } else {
        bos = (long long)n * p.T;
        eos = bos + p.T;
    }

    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *g = static_cast<const Tin *>(p.g);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    Tin *o = static_cast<Tin *>(p.o);

    __shared__ float sk[2][DK], sq[2][DK], sa[2][DK], sv[2][DV], sb[2];
    __shared__ float red_k[2][kWarps][DV], red_q[2][kWarps][DV], red_qk[2][3][kWarps];

    const int row0 = w * RPW, col0 = l * CPL;
    const bool norm = EXT && p.qk_l2norm;
    static_assert(DK == DV, "square states");
    const long long init_off = p.init ? state_slot_offset(p.init_idx, p.pool, n, H, h, DK, p.err) : -1;
    float s[RPW][CPL];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        if (init_off >= 0) {
            load_state<CPL>(p.init + init_off + (size_t)(row0 + r) * DV + col0, s[r]);
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) s[r][c] = 0.f;
        }
    }

    for (long long t = bos; t < eos; ++t) {
        const int buf = (int)((t - bos) & 1);
        const size_t rr = (size_t)t * H + h;
        if (tid < DK) {
            sk[buf][tid] = load_elem(k, rr * DK + tid);
            sq[buf][tid] = load_elem(q, rr * DK + tid);
            float gv = load_elem(g, rr * DK + tid);
            if (p.gate_bound > 0.f) gv = -p.gate_bound / (1.f + expf(-gv));  // scaled sigmoid of a logit
            sa[buf][tid] = expf(gv);
        } else if (tid < DK + DV) {
            sv[buf][tid - DK] = load_elem(v, rr * DV + (tid - DK));
        }
        if (tid == kThreads - 1) sb[buf] = load_elem(beta, rr);
        __syncthreads();

        // Decay the owned rows and form partial column sums of k^T S' and q^T S'.
        float pk[CPL], pq[CPL], pqk = 0.f, pkk = 0.f, pqq = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) pk[c] = pq[c] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float a = sa[buf][row0 + r], kk = sk[buf][row0 + r], qq = sq[buf][row0 + r];
            pqk = fmaf(kk, qq, pqk);
            if (norm) {
                pkk = fmaf(kk, kk, pkk);
                pqq = fmaf(qq, qq, pqq);
            }
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                s[r][c] *= a;
                pk[c] = fmaf(kk, s[r][c], pk[c]);
                pq[c] = fmaf(qq, s[r][c], pq[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            red_k[buf][w][col0 + c] = pk[c];
            red_q[buf][w][col0 + c] = pq[c];
        }
        if (l == 0) {
            red_qk[buf][0][w] = pqk;
            if (norm) {
                red_qk[buf][1][w] = pkk;
                red_qk[buf][2][w] = pqq;
            }
        }
        __syncthreads();

        float qk = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) qk += red_qk[buf][0][i];
        // L2-normalised q and k are q / |q|, k / |k|: every use of k and q is linear in it, so
        // the norms scale the reductions and the write instead of the inputs.
        float nk = 1.f, nq = 1.f;
        if (norm) {
            float kk2 = 0.f, qq2 = 0.f;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) {
                kk2 += red_qk[buf][1][i];
                qq2 += red_qk[buf][2][i];
            }
            nk = rsqrtf(kk2 + 1e-6f);
            nq = rsqrtf(qq2 + 1e-6f);
            qk *= nk * nq;
        }
        const float b = sb[buf];
        float u[CPL], oo[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            float ks = 0.f, qs = 0.f;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) {
                ks += red_k[buf][i][col0 + c];
                qs += red_q[buf][i][col0 + c];
            }
            u[c] = b * (sv[buf][col0 + c] - ks * nk);
            oo[c] = fmaf(qk, u[c], qs * nq);
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float kk = sk[buf][row0 + r] * nk;
#pragma unroll
            for (int c = 0; c < CPL; ++c) s[r][c] = fmaf(kk, u[c], s[r][c]);
        }
        if (w == 0) {
            const Tin *z = EXT ? static_cast<const Tin *>(p.out_gate) : nullptr;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                float ov = oo[c];
                if (z) ov *= 1.f / (1.f + expf(-load_elem(z, rr * DV + col0 + c)));  // output gate sigmoid(z)
                store_elem(o, rr * DV + col0 + c, ov);
            }
        }
    }

    const long long fin_off = p.fin ? state_slot_offset(p.fin_idx, p.pool, n, H, h, DK, p.err) : -1;
    if (fin_off >= 0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            store_state<CPL>(p.fin + fin_off + (size_t)(row0 + r) * DV + col0, s[r]);
    }
}

template <typename Tin>
cudaError_t launch_typed(int d, const RunParams &p, cudaStream_t s) {
    const dim3 grid((unsigned)(p.n_seqs * p.H)), block(kThreads);
    const bool ext = p.qk_l2norm || p.out_gate;
    switch (d * 2 + (ext ? 1 : 0)) {
        case 64: recurrent_kernel<Tin, 32, 32, false><<<grid, block, 0, s>>>(p); break;
        case 65: recurrent_kernel<Tin, 32, 32, true><<<grid, block, 0, s>>>(p); break;
        case 128: recurrent_kernel<Tin, 64, 64, false><<<grid, block, 0, s>>>(p); break;
        case 129: recurrent_kernel<Tin, 64, 64, true><<<grid, block, 0, s>>>(p); break;
        case 256: recurrent_kernel<Tin, 128, 128, false><<<grid, block, 0, s>>>(p); break;
        case 257: recurrent_kernel<Tin, 128, 128, true><<<grid, block, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(kda_dtype dtype, int dk, int dv, const RunParams &p, cudaStream_t s) {
    if (dk != dv) return cudaErrorInvalidValue;
    if ((long long)p.n_seqs * p.H == 0) return cudaSuccess;
    return dtype == KDA_BF16 ? launch_typed<__nv_bfloat16>(dk, p, s) : launch_typed<float>(dk, p, s);
}

}  // namespace kda
