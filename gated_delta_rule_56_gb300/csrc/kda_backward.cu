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
// and each token's state is rebuilt from the nearest of those (at most kSub - 1 steps). A
// chunk's inputs (k, exp g, q as fp32 rows, beta, and v, dO of the CTA's columns) are staged in
// shared memory once per CTA, so every step reads them there. dq, dk, dg and dbeta are sums over
// all columns: per kSub tokens the warps add their parts in shared
// memory, then the CTA adds the block to the fp32 outputs with global atomics (one per column
// block); dv and dS_initial belong to one column and are stored directly.
//
// This kernel serves d_k = d_v in {32, 64}; launch_backward sends d = 128 to the chunkwise
// tensor-core kernel of kda_backward_chunked.cu, which writes every output itself.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kCols = 16;   // value columns (warps) per CTA
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

// Shared-memory layout (bytes) of one staged chunk (kChunk tokens) for head size DK. k and q
// keep the input type (bf16 rows are exact), the decays are stored as exp(g) in fp32.
template <int DK, typename Tin>
struct Stage {
    static constexpr size_t A = 0;                                  // fp32 [kChunk][DK]: exp(g)
    static constexpr size_t V = A + kChunk * DK * 4;                // fp32 [kChunk][kCols]: v of the CTA's columns
    static constexpr size_t DO = V + kChunk * kCols * 4;            // fp32 [kChunk][kCols]: dO of those columns
    static constexpr size_t B = DO + kChunk * kCols * 4;            // fp32 [kChunk]: beta
    static constexpr size_t ACC = B + kChunk * 4;                   // fp32 [kSub][3][DK]: dq, dk, dg sums
    static constexpr size_t ACCB = ACC + kSub * 3 * DK * 4;         // fp32 [kSub]: dbeta sums
    static constexpr size_t K = ACCB + kSub * 4;                    // Tin [kChunk][DK]: k
    static constexpr size_t Q = K + kChunk * DK * sizeof(Tin);      // Tin [kChunk][DK]: q
    static constexpr size_t BYTES = Q + kChunk * DK * sizeof(Tin);
    static_assert(K % 16 == 0 && Q % 16 == 0, "row alignment");
    __device__ static float *f(uint8_t *sm, size_t off) { return reinterpret_cast<float *>(sm + off); }
    __device__ static Tin *t(uint8_t *sm, size_t off) { return reinterpret_cast<Tin *>(sm + off); }
};

// RPL consecutive elements of a staged row, widened to fp32.
template <int RPL>
__device__ __forceinline__ void row_load(const float *p, float (&x)[RPL]) {
#pragma unroll
    for (int i = 0; i < RPL; ++i) x[i] = p[i];
}
template <int RPL>
__device__ __forceinline__ void row_load(const __nv_bfloat16 *p, float (&x)[RPL]) {
#pragma unroll
    for (int i = 0; i < RPL; ++i) x[i] = __bfloat162float(p[i]);
}

// Stage the inputs of tokens [c0, c0 + kChunk) (rows past eos read as identity tokens: k = 0,
// exp g = 1). With `rev` also q and dO, which only the reverse sweep reads.
template <typename Tin, int DK>
__device__ __forceinline__ void stage_chunk(uint8_t *sm, const RunParams &p, const Tin *dop, long long c0,
                                            long long eos, int H, int h, int j0, bool rev) {
    using L = Stage<DK, Tin>;
    const Tin *kp = static_cast<const Tin *>(p.k), *gp = static_cast<const Tin *>(p.g);
    const Tin *qp = static_cast<const Tin *>(p.q), *vp = static_cast<const Tin *>(p.v);
    const Tin *bp = static_cast<const Tin *>(p.beta);
    const Tin zero = Tin(0.f);
    for (int e = threadIdx.x; e < kChunk * DK; e += kThreads) {
        const int t = e / DK, i = e % DK;
        const bool live = c0 + t < eos;
        const size_t r = ((size_t)(c0 + t) * H + h) * DK + i;
        L::t(sm, L::K)[e] = live ? kp[r] : zero;
        L::f(sm, L::A)[e] = live ? expf(ld(gp, r)) : 1.f;
        if (rev) L::t(sm, L::Q)[e] = live ? qp[r] : zero;
    }
    for (int e = threadIdx.x; e < kChunk * kCols; e += kThreads) {
        const int t = e / kCols, c = e % kCols;
        const bool live = c0 + t < eos;
        const size_t r = ((size_t)(c0 + t) * H + h) * DK + j0 + c;
        L::f(sm, L::V)[e] = live ? ld(vp, r) : 0.f;
        if (rev) L::f(sm, L::DO)[e] = live ? ld(dop, r) : 0.f;
    }
    for (int t = threadIdx.x; t < kChunk; t += kThreads)
        L::f(sm, L::B)[t] = c0 + t < eos ? ld(bp, (size_t)(c0 + t) * H + h) : 0.f;
}

// One forward token (index tt of the staged chunk) on the lane's rows of column `col`.
template <typename Tin, int DK, int RPL>
__device__ __forceinline__ void step(float (&S)[RPL], uint8_t *sm, int tt, int row0, int col) {
    using L = Stage<DK, Tin>;
    float k[RPL];
    row_load<RPL>(L::t(sm, L::K) + tt * DK + row0, k);
    const float *a = L::f(sm, L::A) + tt * DK + row0;
    float ks = 0.f;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        S[i] *= a[i];
        ks = fmaf(k[i], S[i], ks);
    }
    const float u = L::f(sm, L::B)[tt] * (L::f(sm, L::V)[tt * kCols + col] - warp_sum(ks));
#pragma unroll
    for (int i = 0; i < RPL; ++i) S[i] = fmaf(k[i], u, S[i]);
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreads, 2) backward_kernel(RunParams p, const void *d_o, const float *d_fin,
                                                          float *dq, float *dk, float *dv, float *dg,
                                                          float *dbeta, float *d_init, float *ck) {
    constexpr int DV = DK, RPL = DK / 32;
    using L = Stage<DK, Tin>;
    extern __shared__ __align__(16) uint8_t sm[];
    float *acc = L::f(sm, L::ACC), *accb = L::f(sm, L::ACCB);
    const int H = p.H, h = blockIdx.x % H, n = blockIdx.x / H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = blockIdx.y * kCols, j = j0 + warp;  // this warp's value column
    const int row0 = lane * RPL;
    const Tin *dop = static_cast<const Tin *>(d_o);

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

    for (int e = threadIdx.x; e < kSub * 3 * DK; e += kThreads) acc[e] = 0.f;
    if (threadIdx.x < kSub) accb[threadIdx.x] = 0.f;

    const size_t sbase = ((size_t)n * H + h) * DK * DV;
    float S[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) S[i] = p.init ? p.init[sbase + (size_t)(row0 + i) * DV + j] : 0.f;

    // Forward sweep: the column state at every chunk start.
    for (int c = 0; c < nchunks; ++c) {
        const long long c0 = bos + (long long)c * kChunk;
        float *dst = ck_ptr(c);
#pragma unroll
        for (int i = 0; i < RPL; ++i) dst[i] = S[i];
        __syncthreads();  // the previous chunk's inputs are no longer read
        stage_chunk<Tin, DK>(sm, p, dop, c0, eos, H, h, j0, false);
        __syncthreads();
        const int nt = (int)min((long long)kChunk, eos - c0);
        for (int tt = 0; tt < nt; ++tt) step<Tin, DK, RPL>(S, sm, tt, row0, warp);
    }

    float dS[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) dS[i] = d_fin ? d_fin[sbase + (size_t)(row0 + i) * DV + j] : 0.f;

    for (int c = nchunks - 1; c >= 0; --c) {
        const long long c0 = bos + (long long)c * kChunk;
        __syncthreads();
        stage_chunk<Tin, DK>(sm, p, dop, c0, eos, H, h, j0, true);
        __syncthreads();
        // Replay the chunk from its checkpoint, keeping the state every kSub tokens.
        float sub[kChunk / kSub][RPL];
        {
            const float *src = ck_ptr(c);
#pragma unroll
            for (int i = 0; i < RPL; ++i) S[i] = src[i];
        }
        const int nt = (int)min((long long)kChunk, eos - c0);
#pragma unroll
        for (int s = 0; s < kChunk / kSub; ++s) {
#pragma unroll
            for (int i = 0; i < RPL; ++i) sub[s][i] = S[i];
            const int t1 = min((s + 1) * kSub, nt);
            for (int tt = s * kSub; tt < t1; ++tt) step<Tin, DK, RPL>(S, sm, tt, row0, warp);
        }
#pragma unroll
        for (int s = kChunk / kSub - 1; s >= 0; --s) {
            const int tb = s * kSub;
            if (tb >= nt) continue;  // uniform over the CTA
            const int te = min(tb + kSub, nt);
            for (int tt = te - 1; tt >= tb; --tt) {
                // The state before token tt, rebuilt from the register checkpoint.
#pragma unroll
                for (int i = 0; i < RPL; ++i) S[i] = sub[s][i];
                for (int u = tb; u < tt; ++u) step<Tin, DK, RPL>(S, sm, u, row0, warp);
                float k[RPL], q[RPL];
                row_load<RPL>(L::t(sm, L::K) + tt * DK + row0, k);
                row_load<RPL>(L::t(sm, L::Q) + tt * DK + row0, q);
                const float *a = L::f(sm, L::A) + tt * DK + row0;
                const float beta = L::f(sm, L::B)[tt], dov = L::f(sm, L::DO)[tt * kCols + warp];
                float Sd[RPL], ks = 0.f;
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    Sd[i] = a[i] * S[i];
                    ks = fmaf(k[i], Sd[i], ks);
                }
                const float w = L::f(sm, L::V)[tt * kCols + warp] - warp_sum(ks), u = beta * w;
                float kd = 0.f;
                const int t_ = tt - tb;
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    atomicAdd(&acc[(t_ * 3 + 0) * DK + row0 + i], fmaf(k[i], u, Sd[i]) * dov);  // dq: S' do
                    dS[i] = fmaf(q[i], dov, dS[i]);
                    kd = fmaf(k[i], dS[i], kd);
                }
                const float du = warp_sum(kd), bdu = beta * du;
                if (lane == 0) {
                    dv[((size_t)(c0 + tt) * H + h) * DV + j] = bdu;
                    atomicAdd(&accb[t_], du * w);
                }
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    atomicAdd(&acc[(t_ * 3 + 1) * DK + row0 + i], dS[i] * u - Sd[i] * bdu);  // dk
                    const float dsd = dS[i] - k[i] * bdu;
                    atomicAdd(&acc[(t_ * 3 + 2) * DK + row0 + i], dsd * Sd[i]);               // dg
                    dS[i] = a[i] * dsd;
                }
            }
            // This block of tokens is complete in shared memory: add it to the outputs.
            __syncthreads();
            const int nb = te - tb;
            for (int e = threadIdx.x; e < kSub * 3 * DK; e += kThreads) {
                const int t_ = e / (3 * DK), which = (e / DK) % 3, i = e % DK;
                if (t_ < nb) {
                    float *out = which == 0 ? dq : (which == 1 ? dk : dg);
                    atomicAdd(out + ((size_t)(c0 + tb + t_) * H + h) * DK + i, acc[e]);
                }
                acc[e] = 0.f;
            }
            if (threadIdx.x < kSub) {
                if ((int)threadIdx.x < nb) atomicAdd(dbeta + (size_t)(c0 + tb + threadIdx.x) * H + h, accb[threadIdx.x]);
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

template <typename Tin, int DK>
cudaError_t launch_dk(const dim3 &grid, const RunParams &p, const void *d_o, const float *d_fin, float *dq,
                      float *dk, float *dv, float *dg, float *dbeta, float *d_init, float *ck, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(backward_kernel<Tin, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Stage<DK, Tin>::BYTES);
    if (e != cudaSuccess) return e;
    backward_kernel<Tin, DK><<<grid, kThreads, Stage<DK, Tin>::BYTES, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_typed(int d, const RunParams &p, const void *d_o, const float *d_fin, float *dq, float *dk,
                         float *dv, float *dg, float *dbeta, float *d_init, float *ck, cudaStream_t s) {
    const dim3 grid((unsigned)(p.n_seqs * p.H), (unsigned)(d / kCols));
    switch (d) {
        case 32: return launch_dk<Tin, 32>(grid, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck, s);
        case 64: return launch_dk<Tin, 64>(grid, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck, s);
        case 128: return launch_dk<Tin, 128>(grid, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t backward_workspace_bytes(int T_total, int n_seqs, int H, int d) {
    if (T_total < 0 || n_seqs < 0 || H <= 0 || d <= 0) return 0;
    if (d == 128) return backward_chunked_workspace_bytes(T_total, n_seqs, H);
    return ((size_t)T_total / kChunk + (size_t)n_seqs + 1) * (size_t)H * d * d * sizeof(float);
}

cudaError_t launch_backward(kda_dtype dtype, int d, const RunParams &p, const void *d_o, const float *d_fin,
                            float *dq, float *dk, float *dv, float *dg, float *dbeta, float *d_init, void *ws,
                            cudaStream_t s) {
    if ((long long)p.n_seqs * p.H == 0) return cudaSuccess;
    if (d == 128)  // chunkwise on 16-token tiles (kda_backward_chunked.cu); writes every output itself
        return launch_backward_chunked(dtype, p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ws, s);
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    const size_t nk = (size_t)rows * p.H * d;
    // dq, dk, dg and dbeta are sums of atomic adds: start them at zero (dv is stored directly).
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaGetLastError();
    const unsigned zb = 4u * (unsigned)sms;  // four 256-thread blocks per SM
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
