// kda_backward.cu -- gradients of the KDA recurrence on CUDA cores.
//
// For L = sum(dO * O) + sum(dS_final * S_final) the call returns dq, dk, dv, dg (w.r.t. the
// log-decay), dbeta and dS_initial, all fp32. The pages train the model ("Kimi K3 Explained",
// researchpapers.dev) but give no gradient method; this is reverse-mode differentiation of the
// token recurrence ("Inside Kimi K3's Architecture", "Kimi Delta Attention: the linear core"):
//     forward  Sd = Diag(a) S,  w = v - Sd^T k,  u = beta w,  S' = Sd + k u^T,  o = S'^T q
//     reverse  dq = S' do;  dS += q do^T;  du = dS^T k;  dk = dS u - Sd (beta du);  dv = beta du;
//              dbeta = du . w;  dSd = dS - k (beta du)^T;  dg = rowsum(dSd * Sd);  dS = Diag(a) dSd
//
// Work split. Every value column j of the state is its own d_k-vector recurrence (the columns
// share k, a, beta, q but nothing else), so one warp carries one column: lane l holds key rows
// [l*RPL, (l+1)*RPL). A CTA of kCols warps takes kCols columns of one (sequence, head), so no
// thread ever needs another column's state. The reverse sweep needs the state before every
// token: a forward sweep stores the column state every kChunk tokens (global workspace); each
// chunk is then replayed from its checkpoint keeping the state every kSub tokens in registers,
// and each token's state is rebuilt from the nearest of those (at most kSub - 1 steps). dq, dk,
// dg and dbeta are sums over all columns: per kSub tokens the warps add their parts in shared
// memory, then the CTA adds the block to the fp32 outputs with global atomics (one per column
// block); dv and dS_initial belong to one column and are stored directly.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kCols = 8;    // value columns (warps) per CTA
constexpr int kChunk = 64;  // tokens between stored checkpoints
constexpr int kSub = 8;     // tokens between register checkpoints
constexpr int kThreads = kCols * 32;

__device__ __forceinline__ float ld(const float *p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Per-token inputs a lane needs: its rows of k (and a = exp g), beta and v of the warp's column.
template <typename Tin, int RPL>
struct Tok {
    float k[RPL], a[RPL], beta, v;
    __device__ __forceinline__ void load(const RunParams &p, size_t r, int row0, int j, int DV) {
        const Tin *kk = static_cast<const Tin *>(p.k) + r * (RPL * 32) + row0;
        const Tin *gg = static_cast<const Tin *>(p.g) + r * (RPL * 32) + row0;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            k[i] = ld(kk, i);
            a[i] = expf(ld(gg, i));
        }
        beta = ld(static_cast<const Tin *>(p.beta), r);
        v = ld(static_cast<const Tin *>(p.v), r * DV + j);
    }
};

// One forward token on the lane's rows of one column.
template <typename Tin, int RPL>
__device__ __forceinline__ void step(float (&S)[RPL], const Tok<Tin, RPL> &t) {
    float ks = 0.f;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        S[i] *= t.a[i];
        ks = fmaf(t.k[i], S[i], ks);
    }
    const float u = t.beta * (t.v - warp_sum(ks));
#pragma unroll
    for (int i = 0; i < RPL; ++i) S[i] = fmaf(t.k[i], u, S[i]);
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreads) backward_kernel(RunParams p, const void *d_o, const float *d_fin,
                                                          float *dq, float *dk, float *dv, float *dg,
                                                          float *dbeta, float *d_init, float *ck) {
    constexpr int DV = DK, RPL = DK / 32;
    __shared__ float acc[kSub][3][DK];  // dq, dk, dg of the current kSub tokens, summed over columns
    __shared__ float accb[kSub];        // dbeta
    const int H = p.H, h = blockIdx.x % H, n = blockIdx.x / H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.y * kCols + warp;  // this warp's value column
    const int row0 = lane * RPL;

    long long bos, eos;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > p.T || (n == 0 && bos != 0) || (n == p.n_seqs - 1 && eos != p.T)) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBadSeqlens);
            return;
        }
    } else {
        bos = (long long)n * p.T;
        eos = bos + p.T;
    }
    // Checkpoint slots of this sequence: [bos / kChunk + n, ...) never overlaps the next sequence's.
    const long long ck0 = bos / kChunk + n;
    const int nchunks = (int)((eos - bos + kChunk - 1) / kChunk);
    auto ck_ptr = [&](int c) { return ck + (((size_t)(ck0 + c) * H + h) * DV + j) * DK + row0; };

    for (int e = threadIdx.x; e < kSub * 3 * DK; e += kThreads) (&acc[0][0][0])[e] = 0.f;
    if (threadIdx.x < kSub) accb[threadIdx.x] = 0.f;

    const size_t sbase = ((size_t)n * H + h) * DK * DV;
    float S[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) S[i] = p.init ? p.init[sbase + (size_t)(row0 + i) * DV + j] : 0.f;

    // Forward sweep: the column state at every chunk start.
    for (int c = 0; c < nchunks; ++c) {
        float *dst = ck_ptr(c);
#pragma unroll
        for (int i = 0; i < RPL; ++i) dst[i] = S[i];
        const long long t1 = min(bos + (long long)(c + 1) * kChunk, eos);
        for (long long t = bos + (long long)c * kChunk; t < t1; ++t) {
            Tok<Tin, RPL> tk;
            tk.load(p, (size_t)t * H + h, row0, j, DV);
            step<Tin, RPL>(S, tk);
        }
    }

    float dS[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) dS[i] = d_fin ? d_fin[sbase + (size_t)(row0 + i) * DV + j] : 0.f;
    __syncthreads();  // accumulators zeroed

    const Tin *qp = static_cast<const Tin *>(p.q);
    const Tin *dop = static_cast<const Tin *>(d_o);
    for (int c = nchunks - 1; c >= 0; --c) {
        const long long c0 = bos + (long long)c * kChunk;
        // Replay the chunk from its checkpoint, keeping the state every kSub tokens.
        float sub[kChunk / kSub][RPL];
        {
            const float *src = ck_ptr(c);
#pragma unroll
            for (int i = 0; i < RPL; ++i) S[i] = src[i];
        }
#pragma unroll
        for (int s = 0; s < kChunk / kSub; ++s) {
#pragma unroll
            for (int i = 0; i < RPL; ++i) sub[s][i] = S[i];
            const long long t1 = min(c0 + (long long)(s + 1) * kSub, eos);
            for (long long t = c0 + (long long)s * kSub; t < t1; ++t) {
                Tok<Tin, RPL> tk;
                tk.load(p, (size_t)t * H + h, row0, j, DV);
                step<Tin, RPL>(S, tk);
            }
        }
#pragma unroll
        for (int s = kChunk / kSub - 1; s >= 0; --s) {
            const long long tb = c0 + (long long)s * kSub;
            if (tb >= eos) continue;  // uniform over the CTA
            const long long te = min(tb + kSub, eos);
            for (long long t = te - 1; t >= tb; --t) {
                // The state before token t, rebuilt from the register checkpoint.
#pragma unroll
                for (int i = 0; i < RPL; ++i) S[i] = sub[s][i];
                for (long long u = tb; u < t; ++u) {
                    Tok<Tin, RPL> tk;
                    tk.load(p, (size_t)u * H + h, row0, j, DV);
                    step<Tin, RPL>(S, tk);
                }
                const size_t r = (size_t)t * H + h;
                Tok<Tin, RPL> tk;
                tk.load(p, r, row0, j, DV);
                const float dov = ld(dop, r * DV + j);
                float q[RPL], Sd[RPL], ks = 0.f;
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    q[i] = ld(qp, r * DK + row0 + i);
                    Sd[i] = tk.a[i] * S[i];
                    ks = fmaf(tk.k[i], Sd[i], ks);
                }
                const float w = tk.v - warp_sum(ks), u = tk.beta * w;
                float kd = 0.f;
                const int tt = (int)(t - tb);
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    atomicAdd(&acc[tt][0][row0 + i], fmaf(tk.k[i], u, Sd[i]) * dov);  // dq: S' do
                    dS[i] = fmaf(q[i], dov, dS[i]);
                    kd = fmaf(tk.k[i], dS[i], kd);
                }
                const float du = warp_sum(kd), bdu = tk.beta * du;
                if (lane == 0) {
                    dv[r * DV + j] = bdu;
                    atomicAdd(&accb[tt], du * w);
                }
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    atomicAdd(&acc[tt][1][row0 + i], dS[i] * u - Sd[i] * bdu);  // dk
                    const float dsd = dS[i] - tk.k[i] * bdu;
                    atomicAdd(&acc[tt][2][row0 + i], dsd * Sd[i]);               // dg
                    dS[i] = tk.a[i] * dsd;
                }
            }
            // This block of tokens is complete in shared memory: add it to the outputs.
            __syncthreads();
            const int nt = (int)(te - tb);
            for (int e = threadIdx.x; e < kSub * 3 * DK; e += kThreads) {
                const int t_ = e / (3 * DK), which = (e / DK) % 3, i = e % DK;
                float *a = &(&acc[0][0][0])[e];
                if (t_ < nt) {
                    float *out = which == 0 ? dq : (which == 1 ? dk : dg);
                    atomicAdd(out + ((size_t)(tb + t_) * H + h) * DK + i, *a);
                }
                *a = 0.f;
            }
            if (threadIdx.x < kSub) {
                if ((int)threadIdx.x < nt) atomicAdd(dbeta + (size_t)(tb + threadIdx.x) * H + h, accb[threadIdx.x]);
                accb[threadIdx.x] = 0.f;
            }
            __syncthreads();
        }
    }
    if (d_init) {
#pragma unroll
        for (int i = 0; i < RPL; ++i) d_init[sbase + (size_t)(row0 + i) * DV + j] = dS[i];
    }
}

__global__ void zero_kernel(float *__restrict__ x, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        x[i] = 0.f;
}

template <typename Tin>
cudaError_t launch_typed(int d, const RunParams &p, const void *d_o, const float *d_fin, float *dq, float *dk,
                         float *dv, float *dg, float *dbeta, float *d_init, float *ck, cudaStream_t s) {
    const dim3 grid((unsigned)(p.n_seqs * p.H), (unsigned)(d / kCols));
    switch (d) {
        case 32: backward_kernel<Tin, 32><<<grid, kThreads, 0, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck); break;
        case 64: backward_kernel<Tin, 64><<<grid, kThreads, 0, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck); break;
        case 128: backward_kernel<Tin, 128><<<grid, kThreads, 0, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_bytes(int T_total, int n_seqs, int H, int d) {
    if (T_total < 0 || n_seqs < 0 || H <= 0 || d <= 0) return 0;
    return ((size_t)T_total / kChunk + (size_t)n_seqs + 1) * (size_t)H * d * d * sizeof(float);
}

cudaError_t launch_backward(kda_dtype dtype, int d, const RunParams &p, const void *d_o, const float *d_fin,
                            float *dq, float *dk, float *dv, float *dg, float *dbeta, float *d_init, void *ws,
                            cudaStream_t s) {
    if ((long long)p.n_seqs * p.H == 0) return cudaSuccess;
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    const size_t nk = (size_t)rows * p.H * d;
    // dq, dk, dg and dbeta are sums of atomic adds: start them at zero (dv is stored directly).
    const unsigned zb = 4 * 152;
    zero_kernel<<<zb, 256, 0, s>>>(dq, nk);
    zero_kernel<<<zb, 256, 0, s>>>(dk, nk);
    zero_kernel<<<zb, 256, 0, s>>>(dg, nk);
    zero_kernel<<<zb, 256, 0, s>>>(dbeta, (size_t)rows * p.H);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    float *ck = static_cast<float *>(ws);
    return dtype == KDA_BF16 ? launch_typed<__nv_bfloat16>(d, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck, s)
                             : launch_typed<float>(d, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck, s);
}

}  // namespace kda
