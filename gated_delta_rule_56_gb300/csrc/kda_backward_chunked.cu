// kda_backward_chunked.cu -- gradients of the KDA recurrence for d_k = d_v = 128, chunkwise.
//
// The same gradients as kda_backward.cu (L = sum(dO * O) + sum(dS_final * S_final); dq, dk, dv,
// dg, dbeta, dS_initial in fp32), computed over chunks of C = 16 tokens in the chunkwise form of
// the recurrence ("Kimi K3 Explained", researchpapers.dev, "Architecture at a glance": the
// chunkwise computation runs on dense tiles). Per chunk, with S the state at its start,
// Gam = cumsum of g over the chunk's rows (per channel), gam = exp(Gam), gC = gam of the last row:
//     Kp = K gam, Km = K / gam, Qp = Q gam, Kc = K gC / gam               (element-wise)
//     Ab = Kp Km^T,  A = strict_lower(Diag(beta) Ab),  X = (I + A)^{-1},  T = X Diag(beta)
//     R = V - Kp S,  U = T R,  P = lower(Qp Km^T),  O = Qp S + P U,  S' = Diag(gC) S + Kc^T U
// and its adjoint, given dO and dS' (the gradient w.r.t. the next chunk's start state):
//     dU = P^T dO + Kc dS',  dR = T^T dU (= dV),  dP = lower(dO U^T),  dT = dU R^T,
//     dX = dT Diag(beta),  dbeta = colsum(X * dT) + rowsum(dA * Ab),  dA = strict_lower(-X^T dX X^T),
//     dQp = dO S^T + dP Km,  dKp = -dR S^T + (Diag(beta) dA) Km,
//     dKm = dP^T Qp + (Diag(beta) dA)^T Kp,  dKc = U dS'^T,  dgC = rowsum(dS' * S),
//     dK = dKp gam + dKm / gam + dKc gC / gam,  dQ = dQp gam,
//     dGam = dKp Kp - dKm Km + dQp Qp - dKc Kc  (+ colsum(dKc Kc) + dgC gC on the last row),
//     dg = reverse cumsum of dGam over the rows,  dS = Qp^T dO - Kp^T dR + Diag(gC) dS'.
// With g >= -5 a 16-row chunk keeps gam and 1/gam within e^{+-80}, inside fp32, so the chunk needs
// no sub-tiling; each exponent is clamped to +-87 so out-of-range gates stay finite.
//
// One CTA of 512 threads per (sequence, head) holds S and dS (fp32, 128 x 128, rows padded to
// 132 floats: 16-byte row reads and the 8-row groups of an ldmatrix are free of bank conflicts,
// fragment reads down a column are 2-way) and the chunk's 16 x 128 tiles in shared memory. Every
// product runs on the tensor cores as warp MMAs (precision per product: see mma3); the triangular
// solve and the element-wise steps run on the CUDA cores in fp32. A forward sweep stores the
// state at every chunk start in the workspace; the reverse sweep reads it back. All columns live
// in one CTA, so every gradient is written directly (no atomics).
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int C = 16;                  // tokens per chunk
constexpr int NT = 512;                // threads per CTA
constexpr int LS = D + 4;              // row stride of S and dS (floats): 16-byte rows, and row i
                                       // starts 33 i 16-byte units in (i mod 8 distinct), so 16-byte
                                       // reads of 8 consecutive rows (an ldmatrix phase) are free of
                                       // bank conflicts; fragment reads down a column (rows t, t + 4
                                       // across 8 columns) are 2-way
constexpr int LT = D + 4;              // row stride of a 16 x 128 tile (floats; 16-byte rows)
constexpr int LM = C + 4;              // row stride of a 16 x 16 matrix (16-byte rows)

// Shared-memory layout (floats).
constexpr int O_S = 0;
constexpr int O_DS = O_S + D * LS;
constexpr int O_GAM = O_DS + D * LS;   // tiles of C x LT
constexpr int O_QP = O_GAM + C * LT;
constexpr int O_KP = O_QP + C * LT;
constexpr int O_KM = O_KP + C * LT;
constexpr int O_R = O_KM + C * LT;     // V, then R = V - Kp S
constexpr int O_U = O_R + C * LT;
constexpr int O_DO = O_U + C * LT;
constexpr int O_DU = O_DO + C * LT;
constexpr int O_DR = O_DU + C * LT;
constexpr int O_DG = O_DR + C * LT;
constexpr int O_AB = O_DG + C * LT;    // 16 x 16 matrices of C x LM
constexpr int O_X = O_AB + C * LM;
constexpr int O_T = O_X + C * LM;
constexpr int O_P = O_T + C * LM;
constexpr int O_DP = O_P + C * LM;
constexpr int O_DT = O_DP + C * LM;
constexpr int O_DAB = O_DT + C * LM;   // Diag(beta) dA
constexpr int O_M = O_DAB + C * LM;    // scratch 16 x 16
constexpr int O_TT = O_M + C * LM;     // T transposed
constexpr int O_BETA = O_TT + C * LM;  // [C]
constexpr int O_DB = O_BETA + C;       // [C] spare (unused; keeps the offsets below)
constexpr int O_GC = O_DB + C;         // [D] gC
constexpr int O_DGC = O_GC + D;        // [D] dgC gC + colsum(dKc Kc)
constexpr int FLOATS = O_DGC + D;
constexpr size_t SMEM = (size_t)FLOATS * sizeof(float);
static_assert(SMEM <= 232448, "shared memory budget");

__device__ __forceinline__ float ld(const float *p, size_t i) { return __ldg(p + i); }

// 16-byte asynchronous copies global -> shared; the thread waits for all of its own with
// cp_async_wait.
__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// The 128-byte lines of rows [t0, t0 + n) of a [rows, H, D] tensor for head h into L2, ahead of
// their use (one line per thread at most; D elements of Tin per row).
template <typename Tin>
__device__ __forceinline__ void prefetch_rows(const Tin *src, long long t0, int n, int H, int h, int slot) {
    constexpr int kLines = D * (int)sizeof(Tin) / 128;  // lines per row
    const int e = (int)threadIdx.x - slot * C * kLines;
    if (e >= 0 && e < n * kLines) {
        const char *a = reinterpret_cast<const char *>(src + ((size_t)(t0 + e / kLines) * H + h) * D) + 128 * (e % kLines);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
}
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }

// gam = exp(cumsum g) per channel over the chunk from the staged g tile (rows past n hold 0),
// gC = its last row.
__device__ __forceinline__ void gate_tile(float *sm, const float *gt) {
    if (threadIdx.x < D) {
        const int i = threadIdx.x;
        float G = 0.f;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            G += gt[r * LT + i];
            sm[O_GAM + r * LT + i] = __expf(fminf(fmaxf(G, -87.f), 87.f));
        }
        sm[O_GC + i] = sm[O_GAM + (C - 1) * LT + i];
    }
}

// Four consecutive elements of a row as floats (one 8-byte load for bf16, 16-byte for fp32).
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xffff0000u));
}
__device__ __forceinline__ float4 ld4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }

// Stage up to five [rows, H, D] tensors' chunk rows [t0, t0 + n) into C x LT tiles (rows past n
// = 0); thread e takes row e / 32, channels 4 (e % 32) .. + 3 of each. Every load of the thread is
// issued before any store, so their latencies overlap.
template <typename Tin, int NTEN>
__device__ __forceinline__ void load_tiles(float *const (&dst)[NTEN], const Tin *const (&src)[NTEN], long long t0,
                                           int n, int H, int h) {
    static_assert(C * D == 4 * NT, "one 4-element group per thread and tensor");
    const int r = threadIdx.x / (D / 4), i = 4 * (threadIdx.x % (D / 4));
    float4 v[NTEN];
#pragma unroll
    for (int a = 0; a < NTEN; ++a)
        v[a] = r < n ? ld4(src[a] + ((size_t)(t0 + r) * H + h) * D + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int a = 0; a < NTEN; ++a) *reinterpret_cast<float4 *>(dst[a] + r * LT + i) = v[a];
}

// ---- products on the tensor cores: warp-level mma.sync m16n8k8 with tf32 operands. With SPLIT = 3
// every fp32 operand x is split into a tf32 high part and the tf32 rounding of the rest, and a
// product is taken as lo*hi + hi*lo + hi*hi (the lo*lo term is below fp32 rounding), so the result
// keeps fp32 accuracy; with SPLIT = 1 a product is the single tf32 one. The 16 x 16 chunk factors
// (Ab, P, dP, dT), U = T R, dR = T^T dU and the finishing products with dP and dAb always take
// SPLIT = 3: they cost little and feed the cancelling sums behind dbeta and dq, whose error single
// tf32 products there raise several times. The products with the 128 x 128 states, and P^T dO
// (which shares its accumulator with Kc dS'), take SPLIT = 3 for fp32 inputs and SPLIT = 1 for
// bf16 inputs (rounded to 2^-9 already, coarser than tf32's 2^-11): gradients then
// agree with the fp64 adjoint to about 3e-4 relative (Frobenius) instead of 2e-6, in three
// quarters of the time.
// Fragment of lane l (g = l / 4, t = l % 4): A (16 x 8) rows g, g + 8 and columns t, t + 4;
// B (8 x 8) rows t, t + 4 and column g; C (16 x 8) rows g, g + 8, columns 2t, 2t + 1.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(x - __uint_as_float(hi)));
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Four 8 x 4 blocks of 32-bit words from shared memory in one instruction: ldmatrix reads 8 x 8
// matrices of 16-bit elements, so lane l gets word (l / 4, l % 4) of each block, which is the
// tf32 fragment layout. Lanes 8m .. 8m + 7 give the addresses of the rows of block m (16-byte
// aligned); r[m] is the lane's word of block m.
__device__ __forceinline__ void ldsm_x4(float (&r)[4], const float *p) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t x0, x1, x2, x3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                 : "r"(a)
                 : "memory");
    r[0] = __uint_as_float(x0);
    r[1] = __uint_as_float(x1);
    r[2] = __uint_as_float(x2);
    r[3] = __uint_as_float(x3);
}

// The lane's row address for A fragments of a 16 x k row-major tile (row stride ld): blocks
// (rows 0-7, columns k..k+3), (rows 8-15, k..k+3), (rows 0-7, k+4..k+7), (rows 8-15, k+4..k+7).
__device__ __forceinline__ const float *a_frag_row(const float *a, int ld) {
    const int lane = threadIdx.x & 31;
    return a + ((lane & 7) + 8 * ((lane >> 3) & 1)) * ld + 4 * (lane >> 4);
}

// The lane's row address for the B fragments of two k steps from an n-major operand (element
// (k, n) at b[n * ld + k]): blocks (rows n0..n0+7, columns k + 4m .. + 3), m = 0..3, give b0, b1
// of step k and b0, b1 of step k + 8.
__device__ __forceinline__ const float *b_frag_row(const float *b, int ld, int n0) {
    const int lane = threadIdx.x & 31;
    return b + (n0 + (lane & 7)) * ld + 4 * (lane >> 3);
}

// c += a b for fp32 fragments a (A layout) and b (B layout).
template <int SPLIT>
__device__ __forceinline__ void mma3(float (&c)[4], const float (&a)[4], const float (&b)[2]) {
    uint32_t ah[4], al[4], bh[2], bl[2];
    if (SPLIT == 3) {
#pragma unroll
        for (int q = 0; q < 4; ++q) split_tf32(a[q], ah[q], al[q]);
#pragma unroll
        for (int q = 0; q < 2; ++q) split_tf32(b[q], bh[q], bl[q]);
        mma_tf32(c, al, bh);
        mma_tf32(c, ah, bl);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(ah[q]) : "f"(a[q]));
#pragma unroll
        for (int q = 0; q < 2; ++q) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(bh[q]) : "f"(b[q]));
    }
    mma_tf32(c, ah, bh);
}

// c (rows g, g + 8 x columns n0 + 2t, + 1 of a 16 x 128 result) = a (16 x 128 tile) B (128 x 128
// at row stride LS), for the warp's 8 columns n0 .. n0 + 7.
template <int SPLIT>
__device__ __forceinline__ void tile_times_state(float (&c)[4], const float *a, const float *B, int n0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float *ap = a_frag_row(a, LT);
    float c2[4] = {0.f, 0.f, 0.f, 0.f};  // odd k steps: two independent MMA chains
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = 0.f;
#pragma unroll 2
    for (int k = 0; k < D; k += 16) {
        float a0[4], a1[4];
        ldsm_x4(a0, ap + k);
        ldsm_x4(a1, ap + k + 8);
        const float b0[2] = {B[(k + t) * LS + n0 + g], B[(k + t + 4) * LS + n0 + g]};
        const float b1[2] = {B[(k + 8 + t) * LS + n0 + g], B[(k + 12 + t) * LS + n0 + g]};
        mma3<SPLIT>(c, a0, b0);
        mma3<SPLIT>(c2, a1, b1);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] += c2[q];
}

// M[r][s] (16 x 16) = sum_i a[r][i] * b[s][i] over the 128 channels, on the tensor cores by the
// two warps w0 and w0 + 1 (one 8-column block each; other warps return at once), at fp32 accuracy.
// Two such products on different warps run side by side.
__device__ __forceinline__ void tile_times_tile_t(float *M, const float *a, const float *b, int w0) {
    const int w = (threadIdx.x >> 5) - w0;
    if (w < 0 || w > 1) return;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, n0 = 8 * w;
    const float *ap = a_frag_row(a, LT), *bp = b_frag_row(b, LT, n0);
    float acc[4][4] = {};  // four independent MMA chains over the k steps
#pragma unroll
    for (int k = 0; k < D; k += 16) {
        float a0[4], a1[4], bb[4];
        ldsm_x4(bb, bp + k);
        ldsm_x4(a0, ap + k);
        ldsm_x4(a1, ap + k + 8);
        const float b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
        const int q = (k >> 3) & 2;
        mma3<3>(acc[q], a0, b0);
        mma3<3>(acc[q + 1], a1, b1);
    }
    float c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = (acc[0][q] + acc[1][q]) + (acc[2][q] + acc[3][q]);
    M[g * LM + n0 + 2 * t] = c[0];
    M[g * LM + n0 + 2 * t + 1] = c[1];
    M[(g + 8) * LM + n0 + 2 * t] = c[2];
    M[(g + 8) * LM + n0 + 2 * t + 1] = c[3];
}

// The chunk's gate products and triangular factors: Kp, Km, Kc (into the tile `kc`), (Qp), Ab,
// A -> X, T (and T transposed), (P).
__device__ __forceinline__ void chunk_factors(float *sm, const float *K, float *kc, bool with_q) {
    {  // thread: row e / 32, channels 4 (e % 32) .. + 3
        const int r = threadIdx.x / (D / 4), i = 4 * (threadIdx.x % (D / 4)), o = r * LT + i;
        const float4 gm = *reinterpret_cast<const float4 *>(sm + O_GAM + o);
        const float4 k = *reinterpret_cast<const float4 *>(K + o);
        const float4 gc = *reinterpret_cast<const float4 *>(sm + O_GC + i);
        const float4 km = make_float4(__fdividef(k.x, gm.x), __fdividef(k.y, gm.y), __fdividef(k.z, gm.z),
                                      __fdividef(k.w, gm.w));
        *reinterpret_cast<float4 *>(sm + O_KP + o) = make_float4(k.x * gm.x, k.y * gm.y, k.z * gm.z, k.w * gm.w);
        *reinterpret_cast<float4 *>(sm + O_KM + o) = km;
        *reinterpret_cast<float4 *>(kc + o) = make_float4(km.x * gc.x, km.y * gc.y, km.z * gc.z, km.w * gc.w);
        if (with_q) {  // Q was loaded into the Qp tile
            float4 *qp = reinterpret_cast<float4 *>(sm + O_QP + o);
            const float4 q = *qp;
            *qp = make_float4(q.x * gm.x, q.y * gm.y, q.z * gm.z, q.w * gm.w);
        }
    }
    __syncthreads();
    tile_times_tile_t(sm + O_AB, sm + O_KP, sm + O_KM, 0);
    if (with_q) tile_times_tile_t(sm + O_P, sm + O_QP, sm + O_KM, 2);
    __syncthreads();
    // X = (I + A)^{-1} for the unit lower-triangular I + A, A = strict_lower(Diag(beta) Ab), by
    // warp 0 in 8 x 8 blocks: the diagonal blocks X11, X22 by forward substitution (lane j < 16:
    // column j of its block), then X21 = -X22 (A21 X11) as two 8 x 8 products (two entries per
    // lane, A21 X11 in the M scratch), X12 = 0; then T = X Diag(beta) and its transpose.
    static_assert(C == 16, "the blocked solve is written for 16-row chunks");
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        if (lane < C) {
            const int j = lane, b0 = lane & 8;
            float x[8];
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const int i = b0 + ii;
                float v = (i == j) ? 1.f : 0.f;
                if (i > j) {
                    const float bi = sm[O_BETA + i];
#pragma unroll
                    for (int kk = 0; kk < ii; ++kk)
                        if (b0 + kk >= j) v = fmaf(-bi * sm[O_AB + i * LM + b0 + kk], x[kk], v);
                }
                x[ii] = v;
            }
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) sm[O_X + (b0 + ii) * LM + j] = x[ii];
        }
        __syncwarp();
        const int i = 8 + (lane >> 2), j0 = 2 * (lane & 3);  // rows 8..15, columns j0, j0 + 1 of 0..7
        {
            const float bi = sm[O_BETA + i];
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float a = bi * sm[O_AB + i * LM + k];
                y0 = fmaf(a, sm[O_X + k * LM + j0], y0);
                y1 = fmaf(a, sm[O_X + k * LM + j0 + 1], y1);
            }
            sm[O_M + i * LM + j0] = y0;
            sm[O_M + i * LM + j0 + 1] = y1;
        }
        __syncwarp();
        {
            float z0 = 0.f, z1 = 0.f;
#pragma unroll
            for (int k = 8; k < C; ++k) {
                const float xk = sm[O_X + i * LM + k];
                z0 = fmaf(xk, sm[O_M + k * LM + j0], z0);
                z1 = fmaf(xk, sm[O_M + k * LM + j0 + 1], z1);
            }
            sm[O_X + i * LM + j0] = -z0;
            sm[O_X + i * LM + j0 + 1] = -z1;
            sm[O_X + (i - 8) * LM + 8 + j0] = 0.f;
            sm[O_X + (i - 8) * LM + 8 + j0 + 1] = 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int e = lane; e < C * C; e += 32) {
            const int r = e / C, c2 = e % C;
            const float x = sm[O_X + r * LM + c2] * sm[O_BETA + c2];
            sm[O_T + r * LM + c2] = x;
            sm[O_TT + c2 * LM + r] = x;
        }
    }
    if (with_q) {  // P = lower(Qp Km^T)
        for (int e = threadIdx.x; e < C * C; e += NT) {
            const int r = e / C, s = e % C;
            if (s > r) sm[O_P + r * LM + s] = 0.f;
        }
    }
    __syncthreads();
}

// Elements (row, n0 + 2t) and (row, n0 + 2t + 1) of a 16 x 128 tile as one 8-byte pair: the
// lane's half of a C fragment row (row g or g + 8).
__device__ __forceinline__ float2 *frag_pair(float *tile, int row, int n0) {
    const int t = threadIdx.x & 3;
    return reinterpret_cast<float2 *>(tile + row * LT + n0 + 2 * t);
}

// c += M B[:, n0 .. n0 + 7] (TRANS: c += M^T B[:, n0 .. n0 + 7]) for a 16 x 16 matrix M (row
// stride LM) and a 16 x 128 tile B, at fp32 accuracy (3xtf32).
template <bool TRANS>
__device__ __forceinline__ void small_times_tile_acc(float (&c)[4], const float *M, const float *B, int n0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float *ap = a_frag_row(M, LM);
#pragma unroll
    for (int k = 0; k < C; k += 8) {
        float af[4];
        if (TRANS) {
            af[0] = M[(k + t) * LM + g];
            af[1] = M[(k + t) * LM + g + 8];
            af[2] = M[(k + t + 4) * LM + g];
            af[3] = M[(k + t + 4) * LM + g + 8];
        } else {
            ldsm_x4(af, ap + k);
        }
        const float bf[2] = {B[(k + t) * LT + n0 + g], B[(k + t + 4) * LT + n0 + g]};
        mma3<3>(c, af, bf);
    }
}

// c = M B[:, n0 .. n0 + 7], as above.
__device__ __forceinline__ void small_times_tile(float (&c)[4], const float *M, const float *B, int n0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = 0.f;
    small_times_tile_acc<false>(c, M, B, n0);
}

// R = V - Kp S (in the R tile, which holds V), then U = T R; warp w takes columns 8 w .. + 7 of
// both, so U needs only the warp's own R columns.
template <int SPLIT>
__device__ __forceinline__ void chunk_u(float *sm) {
    const int g = (threadIdx.x & 31) >> 2, n0 = 8 * (threadIdx.x >> 5);
    float c[4];
    tile_times_state<SPLIT>(c, sm + O_KP, sm + O_S, n0);
    float2 *r0 = frag_pair(sm + O_R, g, n0), *r8 = frag_pair(sm + O_R, g + 8, n0);
    const float2 x0 = *r0, x8 = *r8;
    *r0 = make_float2(x0.x - c[0], x0.y - c[1]);
    *r8 = make_float2(x8.x - c[2], x8.y - c[3]);
    __syncwarp();
    small_times_tile(c, sm + O_T, sm + O_R, n0);
    *frag_pair(sm + O_U, g, n0) = make_float2(c[0], c[1]);
    *frag_pair(sm + O_U, g + 8, n0) = make_float2(c[2], c[3]);
    __syncthreads();
}

// X (128 x 128, row stride LS) <- Diag(gC) X + A1^T B1 + s2 A2^T B2 for 16 x 128 tiles A1, B1, A2,
// B2 (A2 may be null). Warp w takes rows 16 (w / 2) .. + 15 and columns 64 (w % 2) .. + 63; every
// element of X is read and written by the one thread holding it.
template <int SPLIT>
__device__ __forceinline__ void state_update(float *X, const float *gc, const float *A1, const float *B1,
                                             const float *A2, const float *B2, float s2) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int m0 = 16 * (w >> 1), nb0 = 64 * (w & 1);
    float af1[2][4], af2[2][4];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // the A fragments (k = token rows 8 ks ..) of this row block
        const int k = 8 * ks;
        af1[ks][0] = A1[(k + t) * LT + m0 + g];
        af1[ks][1] = A1[(k + t) * LT + m0 + g + 8];
        af1[ks][2] = A1[(k + t + 4) * LT + m0 + g];
        af1[ks][3] = A1[(k + t + 4) * LT + m0 + g + 8];
        if (A2) {
            af2[ks][0] = s2 * A2[(k + t) * LT + m0 + g];
            af2[ks][1] = s2 * A2[(k + t) * LT + m0 + g + 8];
            af2[ks][2] = s2 * A2[(k + t + 4) * LT + m0 + g];
            af2[ks][3] = s2 * A2[(k + t + 4) * LT + m0 + g + 8];
        }
    }
    const float g0 = gc[m0 + g], g8 = gc[m0 + g + 8];
#pragma unroll 2
    for (int nb = 0; nb < 64; nb += 8) {
        const int n = nb0 + nb;
        float2 *x0 = reinterpret_cast<float2 *>(X + (m0 + g) * LS + n + 2 * t);
        float2 *x8 = reinterpret_cast<float2 *>(X + (m0 + g + 8) * LS + n + 2 * t);
        const float2 v0 = *x0, v8 = *x8;
        float c[4] = {v0.x * g0, v0.y * g0, v8.x * g8, v8.y * g8};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k = 8 * ks;
            const float b1[2] = {B1[(k + t) * LT + n + g], B1[(k + t + 4) * LT + n + g]};
            mma3<SPLIT>(c, af1[ks], b1);
            if (A2) {
                const float b2[2] = {B2[(k + t) * LT + n + g], B2[(k + t + 4) * LT + n + g]};
                mma3<SPLIT>(c, af2[ks], b2);
            }
        }
        *x0 = make_float2(c[0], c[1]);
        *x8 = make_float2(c[2], c[3]);
    }
}

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) backward_chunked_kernel(RunParams p, const void *d_o, const float *d_fin,
                                                                 float *dq, float *dk, float *dv, float *dg,
                                                                 float *dbeta, float *d_init, float *ck) {
    constexpr int SPLIT = sizeof(Tin) == 4 ? 3 : 1;  // products at the precision class of the inputs
    extern __shared__ float sm[];
    const int H = p.H, h = blockIdx.x % H, n = blockIdx.x / H, tid = threadIdx.x;
    long long bos, eos;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > p.T || (n == 0 && bos != 0) || (n == p.n_seqs - 1 && eos != p.T)) {
            if (tid == 0) atomicOr(p.err, kErrBadSeqlens);
            return;
        }
    } else {
        bos = (long long)n * p.T;
        eos = bos + p.T;
    }
    const int nc = (int)((eos - bos + C - 1) / C);
    const long long ck0 = bos / C + n;  // this sequence's checkpoint slots (never overlap the next's)
    auto ck_at = [&](int c) { return ck + ((size_t)(ck0 + c) * H + h) * D * D; };
    const Tin *Kg = static_cast<const Tin *>(p.k), *Qg = static_cast<const Tin *>(p.q);
    const Tin *Vg = static_cast<const Tin *>(p.v), *Gg = static_cast<const Tin *>(p.g);
    const Tin *Bg = static_cast<const Tin *>(p.beta), *DOg = static_cast<const Tin *>(d_o);
    const size_t sbase = ((size_t)n * H + h) * D * D;
    float *S = sm + O_S, *dS = sm + O_DS;

    for (int e = tid; e < D * D; e += NT) S[(e / D) * LS + e % D] = p.init ? p.init[sbase + e] : 0.f;
    __syncthreads();

    // ---- forward sweep: the state at every chunk start into the workspace ----------------------
    for (int c = 0; c < nc; ++c) {
        const long long t0 = bos + (long long)c * C;
        const int len = (int)min((long long)C, eos - t0);
        float *dst = ck_at(c);
        for (int e = 4 * tid; e < D * D; e += 4 * NT)
            *reinterpret_cast<float4 *>(dst + e) = *reinterpret_cast<const float4 *>(S + (e / D) * LS + e % D);
        if (c + 1 < nc) {  // the next chunk's rows into L2
            const long long t1 = t0 + C;
            const int l1 = (int)min((long long)C, eos - t1);
            prefetch_rows(Kg, t1, l1, H, h, 0);
            prefetch_rows(Vg, t1, l1, H, h, 1);
            prefetch_rows(Gg, t1, l1, H, h, 2);
        }
        {  // K in the dU tile and g in the dG tile (both free in the forward sweep), V in the R tile
            float *const dst[3] = {sm + O_DU, sm + O_R, sm + O_DG};
            const Tin *const src[3] = {Kg, Vg, Gg};
            load_tiles<Tin, 3>(dst, src, t0, len, H, h);
        }
        if (tid < C) sm[O_BETA + tid] = tid < len ? ld(Bg, (size_t)(t0 + tid) * H + h) : 0.f;
        __syncthreads();
        gate_tile(sm, sm + O_DG);
        __syncthreads();
        chunk_factors(sm, sm + O_DU, sm + O_DR, false);
        chunk_u<SPLIT>(sm);
        // S <- Diag(gC) S + Kc^T U (Kc in the dR tile)
        state_update<SPLIT>(S, sm + O_GC, sm + O_DR, sm + O_U, nullptr, nullptr, 1.f);
        __syncthreads();
    }

    // ---- reverse sweep ---------------------------------------------------------------------------
    for (int e = tid; e < D * D; e += NT) dS[(e / D) * LS + e % D] = d_fin ? d_fin[sbase + e] : 0.f;
    for (int c = nc - 1; c >= 0; --c) {
        const long long t0 = bos + (long long)c * C;
        const int len = (int)min((long long)C, eos - t0);
        __syncthreads();
        if (c == nc - 1) {  // later chunks' start states arrive by cp.async during the chunk after them
            const float *src = ck_at(c);
            for (int e = tid; e < D * D; e += NT) S[(e / D) * LS + e % D] = src[e];
        } else {
            cp_async_wait();
        }
        if (c > 0) {  // the previous chunk's rows into L2
            const long long tp = t0 - C;
            prefetch_rows(Kg, tp, C, H, h, 0);
            prefetch_rows(Qg, tp, C, H, h, 1);
            prefetch_rows(Vg, tp, C, H, h, 2);
            prefetch_rows(DOg, tp, C, H, h, 3);
            prefetch_rows(Gg, tp, C, H, h, 4);
        }
        {  // K in the dU tile until the factors are formed, g in the dG tile until gam is formed
            float *const dst[5] = {sm + O_DU, sm + O_QP, sm + O_R, sm + O_DO, sm + O_DG};
            const Tin *const src[5] = {Kg, Qg, Vg, DOg, Gg};
            load_tiles<Tin, 5>(dst, src, t0, len, H, h);
        }
        if (tid < C) sm[O_BETA + tid] = tid < len ? ld(Bg, (size_t)(t0 + tid) * H + h) : 0.f;
        if (tid < D) sm[O_DGC + tid] = 0.f;
        __syncthreads();
        gate_tile(sm, sm + O_DG);
        __syncthreads();
        chunk_factors(sm, sm + O_DU, sm + O_DG, true);  // Kc in the dG tile until dGam is formed
        chunk_u<SPLIT>(sm);
        // dU = Kc dS + P^T dO (warp w: columns 8 w .. + 7)
        {
            const int lane = tid & 31, g = lane >> 2, t = lane & 3, n0 = 8 * (tid >> 5);
            float c[4];
            tile_times_state<SPLIT>(c, sm + O_DG, dS, n0);
#pragma unroll
            for (int k = 0; k < C; k += 8) {  // P^T (16 x 16) dO (16 x 128)
                const float af[4] = {sm[O_P + (k + t) * LM + g], sm[O_P + (k + t) * LM + g + 8],
                                     sm[O_P + (k + t + 4) * LM + g], sm[O_P + (k + t + 4) * LM + g + 8]};
                const float bf[2] = {sm[O_DO + (k + t) * LT + n0 + g], sm[O_DO + (k + t + 4) * LT + n0 + g]};
                mma3<SPLIT>(c, af, bf);
            }
            *frag_pair(sm + O_DU, g, n0) = make_float2(c[0], c[1]);
            *frag_pair(sm + O_DU, g + 8, n0) = make_float2(c[2], c[3]);
            __syncwarp();
            // dR = T^T dU (= dV, stored) on the warp's own columns of dU; T^T is kept in the Tt matrix
            small_times_tile(c, sm + O_TT, sm + O_DU, n0);
            *frag_pair(sm + O_DR, g, n0) = make_float2(c[0], c[1]);
            *frag_pair(sm + O_DR, g + 8, n0) = make_float2(c[2], c[3]);
            if (g < len) *reinterpret_cast<float2 *>(dv + ((size_t)(t0 + g) * H + h) * D + n0 + 2 * t) = make_float2(c[0], c[1]);
            if (g + 8 < len)
                *reinterpret_cast<float2 *>(dv + ((size_t)(t0 + g + 8) * H + h) * D + n0 + 2 * t) = make_float2(c[2], c[3]);
        }
        __syncthreads();
        // dP = lower(dO U^T), dT = dU R^T
        tile_times_tile_t(sm + O_DP, sm + O_DO, sm + O_U, 4);  // on warps 4-5 and 6-7
        tile_times_tile_t(sm + O_DT, sm + O_DU, sm + O_R, 6);
        __syncthreads();
        // dX = dT Diag(beta); dbeta = colsum(X * dT) + rowsum(dA * Ab); dA = strict_lower(-X^T dX X^T)
        if (tid < C * C) {  // M = dX X^T
            const int r = tid / C, s = tid % C;
            float x = 0.f;
#pragma unroll
            for (int k = 0; k < C; ++k) x = fmaf(sm[O_DT + r * LM + k] * sm[O_BETA + k], sm[O_X + s * LM + k], x);
            sm[O_M + r * LM + s] = x;
            if (s > r) sm[O_DP + r * LM + s] = 0.f;  // dP = lower(dO U^T)
        }
        __syncthreads();
        if (tid < C * C) {  // dAb = Diag(beta) strict_lower(-X^T M)
            const int r = tid / C, s = tid % C;
            float x = 0.f;
#pragma unroll
            for (int k = 0; k < C; ++k) x = fmaf(sm[O_X + k * LM + r], sm[O_M + k * LM + s], x);
            const float da = s < r ? -x : 0.f;
            sm[O_DAB + r * LM + s] = da * sm[O_BETA + r];
            sm[O_P + r * LM + s] = da * sm[O_AB + r * LM + s];  // dA * Ab (P is no longer needed)
        }
        __syncthreads();
        if (tid < C) {
            const int j = tid;
            float x = 0.f;
#pragma unroll
            for (int i = 0; i < C; ++i) x = fmaf(sm[O_X + i * LM + j], sm[O_DT + i * LM + j], x);
#pragma unroll
            for (int s = 0; s < C; ++s) x += sm[O_P + j * LM + s];
            if (j < len) dbeta[(size_t)(t0 + j) * H + h] = x;
        }
        // dO S^T, dR S^T and U dS^T (16 x 128 each; warp w: channels 8 w .. + 7), then, with S and
        // dS read no more, into the R, dU and U tiles.
        {
            const int lane = tid & 31, g = lane >> 2, t = lane & 3, n0 = 8 * (tid >> 5);
            float cq[4] = {0.f, 0.f, 0.f, 0.f}, ckp[4] = {0.f, 0.f, 0.f, 0.f}, cc[4] = {0.f, 0.f, 0.f, 0.f};
            const float *pO = a_frag_row(sm + O_DO, LT), *pR = a_frag_row(sm + O_DR, LT);
            const float *pU = a_frag_row(sm + O_U, LT);
            const float *pS = b_frag_row(S, LS, n0), *pD = b_frag_row(dS, LS, n0);
            float dgc = 0.f;  // sum_j dS[n0 + g][j] S[n0 + g][j] over the lane's columns j = t (mod 4)
#pragma unroll 1
            for (int k = 0; k < D; k += 16) {
                float bs4[4], bd4[4];
                ldsm_x4(bs4, pS + k);
                ldsm_x4(bd4, pD + k);
#pragma unroll
                for (int m = 0; m < 4; ++m) dgc = fmaf(bd4[m], bs4[m], dgc);
#pragma unroll
                for (int hk = 0; hk < 2; ++hk) {
                    const int kk = k + 8 * hk;
                    float ao[4], ar[4], au[4];
                    ldsm_x4(ao, pO + kk);
                    ldsm_x4(ar, pR + kk);
                    ldsm_x4(au, pU + kk);
                    const float bs[2] = {bs4[2 * hk], bs4[2 * hk + 1]}, bd[2] = {bd4[2 * hk], bd4[2 * hk + 1]};
                    mma3<SPLIT>(cq, ao, bs);
                    mma3<SPLIT>(ckp, ar, bs);
                    mma3<SPLIT>(cc, au, bd);
                }
            }
            dgc += __shfl_xor_sync(0xffffffffu, dgc, 1);  // over the 4 lanes t of row n0 + g
            dgc += __shfl_xor_sync(0xffffffffu, dgc, 2);
            if (t == 0) sm[O_DGC + n0 + g] += dgc * sm[O_GC + n0 + g];  // the warp's own channels
            __syncthreads();  // every warp is done with dO, dR and U as operands
            float *T1 = sm + O_R, *T2 = sm + O_DU, *T3 = sm + O_U;
            const int e0 = g * LT + n0 + 2 * t, e8 = (g + 8) * LT + n0 + 2 * t;
            *reinterpret_cast<float2 *>(T1 + e0) = make_float2(cq[0], cq[1]);
            *reinterpret_cast<float2 *>(T1 + e8) = make_float2(cq[2], cq[3]);
            *reinterpret_cast<float2 *>(T2 + e0) = make_float2(ckp[0], ckp[1]);
            *reinterpret_cast<float2 *>(T2 + e8) = make_float2(ckp[2], ckp[3]);
            *reinterpret_cast<float2 *>(T3 + e0) = make_float2(cc[0], cc[1]);
            *reinterpret_cast<float2 *>(T3 + e8) = make_float2(cc[2], cc[3]);
        }
        __syncthreads();
        if (c > 0) {  // S is read no more in this chunk: fetch the previous chunk's start state
            const float *src = ck_at(c - 1);
            for (int e = 4 * tid; e < D * D; e += 4 * NT) cp_async16(S + (e / D) * LS + e % D, src + e);
        }
        // Per (r, i): dQp = dO S^T + dP Km, dKp = -dR S^T + dAb Km, dKm = dP^T Qp + dAb^T Kp and dKc
        // (= U dS^T) -> dq, dk and dGam. Warp w takes channels 8 w .. + 7 in the fragment layout
        // (rows g, g + 8; channels 2t, 2t + 1 of the block); the products as 3xtf32 MMAs.
        {
            const int lane = tid & 31, g = lane >> 2, t = lane & 3, n0 = 8 * (tid >> 5), i0 = n0 + 2 * t;
            float cq[4], ckp[4], ckm[4] = {0.f, 0.f, 0.f, 0.f};
            small_times_tile(cq, sm + O_DP, sm + O_KM, n0);
            small_times_tile(ckp, sm + O_DAB, sm + O_KM, n0);
            small_times_tile_acc<true>(ckm, sm + O_DP, sm + O_QP, n0);
            small_times_tile_acc<true>(ckm, sm + O_DAB, sm + O_KP, n0);
            const float2 gc = *reinterpret_cast<const float2 *>(sm + O_GC + i0);
            float cs[2] = {0.f, 0.f};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = g + 8 * hh;
                const float2 dq2 = *frag_pair(sm + O_R, r, n0), dk2 = *frag_pair(sm + O_DU, r, n0);
                const float2 dc2 = *frag_pair(sm + O_U, r, n0), gm2 = *frag_pair(sm + O_GAM, r, n0);
                const float2 kp2 = *frag_pair(sm + O_KP, r, n0), km2 = *frag_pair(sm + O_KM, r, n0);
                const float2 qp2 = *frag_pair(sm + O_QP, r, n0);
                const float dqa[2] = {dq2.x, dq2.y}, dka[2] = {dk2.x, dk2.y}, dca[2] = {dc2.x, dc2.y};
                const float gma[2] = {gm2.x, gm2.y}, kpa[2] = {kp2.x, kp2.y}, kma[2] = {km2.x, km2.y};
                const float qpa[2] = {qp2.x, qp2.y}, gca[2] = {gc.x, gc.y};
                float dgo[2], dqo[2], dko[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float dqp = dqa[u] + cq[2 * hh + u], dkp = ckp[2 * hh + u] - dka[u];
                    const float dkm = ckm[2 * hh + u], gm = gma[u], gcu = gca[u];
                    const float kc = kma[u] * gcu, dkc = dca[u];
                    dko[u] = dkp * gm + __fdividef(dkm, gm) + dkc * __fdividef(gcu, gm);
                    dqo[u] = dqp * gm;
                    dgo[u] = dkp * kpa[u] - dkm * kma[u] + dqp * qpa[u] - dkc * kc;
                    cs[u] = fmaf(dkc, kc, cs[u]);
                }
                *frag_pair(sm + O_DG, r, n0) = make_float2(dgo[0], dgo[1]);
                if (r < len) {
                    const size_t o = ((size_t)(t0 + r) * H + h) * D + i0;
                    *reinterpret_cast<float2 *>(dq + o) = make_float2(dqo[0], dqo[1]);
                    *reinterpret_cast<float2 *>(dk + o) = make_float2(dko[0], dko[1]);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // sum over the 8 row lanes g of each channel
                cs[u] += __shfl_xor_sync(0xffffffffu, cs[u], 4);
                cs[u] += __shfl_xor_sync(0xffffffffu, cs[u], 8);
                cs[u] += __shfl_xor_sync(0xffffffffu, cs[u], 16);
            }
            if (g == 0) {  // the warp owns these channels: no other writer now
                sm[O_DGC + i0] += cs[0];
                sm[O_DGC + i0 + 1] += cs[1];
            }
        }
        __syncthreads();
        // dg = reverse cumsum of dGam over the chunk's rows (the last row of the chunk, len - 1 for
        // a short final chunk, also takes the gC terms).
        if (tid < D) {
            const int i = tid;
            float acc = sm[O_DGC + i];
            for (int r = C - 1; r >= 0; --r) {
                if (r < len) {
                    acc += sm[O_DG + r * LT + i];
                    dg[((size_t)(t0 + r) * H + h) * D + i] = acc;
                }
            }
        }
        // dS <- Diag(gC) dS + Qp^T dO - Kp^T dR (it reads none of what the dg sums read or write)
        state_update<SPLIT>(dS, sm + O_GC, sm + O_QP, sm + O_DO, sm + O_KP, sm + O_DR, -1.f);
    }
    __syncthreads();
    if (d_init)
        for (int e = tid; e < D * D; e += NT) d_init[sbase + e] = dS[(e / D) * LS + e % D];
}

}  // namespace

size_t backward_chunked_workspace_bytes(int T_total, int n_seqs, int H) {
    if (T_total < 0 || n_seqs < 0 || H <= 0) return 0;
    return ((size_t)T_total / C + (size_t)n_seqs + 1) * (size_t)H * D * D * sizeof(float);
}

cudaError_t launch_backward_chunked(kda_dtype dtype, const RunParams &p, const void *d_o, const float *d_fin,
                                    float *dq, float *dk, float *dv, float *dg, float *dbeta, float *d_init,
                                    void *ws, cudaStream_t s) {
    if ((long long)p.n_seqs * p.H == 0) return cudaSuccess;
    const dim3 grid((unsigned)(p.n_seqs * p.H));
    float *ck = static_cast<float *>(ws);
    cudaError_t e;
    if (dtype == KDA_BF16) {
        e = cudaFuncSetAttribute(backward_chunked_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM);
        if (e != cudaSuccess) return e;
        backward_chunked_kernel<__nv_bfloat16><<<grid, NT, SMEM, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck);
    } else {
        e = cudaFuncSetAttribute(backward_chunked_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
        if (e != cudaSuccess) return e;
        backward_chunked_kernel<float><<<grid, NT, SMEM, s>>>(p, d_o, d_fin, dq, dk, dv, dg, dbeta, d_init, ck);
    }
    return cudaGetLastError();
}

}  // namespace kda
