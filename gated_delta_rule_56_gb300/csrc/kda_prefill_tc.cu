// kda_prefill_tc.cu -- chunked KDA prefill on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// What is computed: the KDA recurrence of "Kimi Delta Attention: the linear core" (maidul-haque
// blog) -- per-channel decay, delta correction, write, read-out -- over chunks of C = 64 tokens,
// in the chunkwise form the pages point to ("Kimi K3 Explained", researchpapers.dev,
// "Architecture at a glance": with the log-decay bounded below, every causal tile of the
// chunkwise computation is a dense tensor-core matmul). Per chunk, with S the d_k x d_v state at
// the chunk start, Gam_r = sum_{s<=r} g_s (per key channel) and gam = exp(Gam):
//     A = strict_lower(Diag(beta) (K*gam)(K/gam)^T),  P = lower((Q*gam)(K/gam)^T)
//     T = (I + A)^{-1} Diag(beta)
//     U = T (V - (K*gam) S)                     (the delta corrections of the chunk)
//     O = (Q*gam) S + P U
//     S <- Diag(gam_last) S + (K*gam_last/gam)^T U
// This equals the token recurrence exactly (unroll it inside the chunk: every intermediate
// state is Diag(gam_t) S plus decayed rank-1 terms k_s u_s^T).
//
// Exponent range. exp(-Gam) reaches e^{320} over a chunk at the decay bound g >= -5, beyond
// fp32/bf16. A and P are therefore built from three 32 x 32 tiles whose factors stay in range:
// the two diagonal half-chunk tiles use the half's middle row (Gam_15, Gam_47) as reference
// (factors within e^{+-80}), and the off-diagonal tile (rows 32..63, columns 0..31) uses the
// boundary row Gam_31, where both factors are <= 1. Every other decay factor is a product of
// in-range terms that are <= 1, so any underflow only drops contributions below 1e-38.
//
// Layout of the work: one CTA of 256 threads per (sequence, head); chunks run in order.
//   TMA: q, k, g tiles (64 rows x 128 channels, 128-byte swizzle) for the next chunk are in
//        flight while the current one computes; the v tile is fetched once the intra-chunk
//        tiles have retired (into their operand region); beta uses plain loads.
//   TMEM (512 columns): [0,64) diagonal A|P tile, [64,96) off-diagonal tile, [96,128) the
//        bf16 A operand -(K+ S)^T then U^T, [128,256) (K+ S | Q+ S -> O), [256,320) U,
//        [320,448) the fp32 state S^T (lanes = d_v), [448,512) its bf16 copy (MMA1's A).
//   MMAs (kind::f16, bf16 operands, fp32 accumulate, M = 128; "tmem" = A read from TMEM):
//        diag  [K*f ; Q*f] x [K/f]^T              N = 64, K = 128
//        off   [K*e ; Q*e] x [K*e']^T             N = 32, K = 128
//        MMA1  S^T (tmem) x [K+ ; Q+]^T           N = 128, K = 128   -> (K+ S)^T, (Q+ S)^T
//        MMA2  V^T x T^T  (V tile, MN-major)      N = 64,  K = 64    -> then += -(K+ S)^T (tmem) x T^T = U^T
//        MMA3  U^T (tmem) x P^T  (onto (Q+ S)^T)  N = 64,  K = 64    -> O^T
//        MMA4  U^T (tmem) x Khat  (MN-major B)    N = 128, K = 64    -> S^T
//   The 64 x 64 triangular inverse: 16 x 16 diagonal blocks by forward substitution on CUDA
//   cores, then the 16->32 and 32->64 block merges as tf32 warp-level MMAs.
// Every mbarrier wait is bounded; on time-out the CTA records kErrTimeout, drains what it
// issued (again bounded), frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;     // chunk length
constexpr int D = 128;    // d_k == d_v
constexpr int NT = 256;   // compute threads (warps 0..7)
constexpr int kIssuer = NT / 32;  // warp 8 issues every MMA and TMA copy
constexpr int NTHREADS = NT + 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr uint32_t SM_Q = 0, SM_K = 16384, SM_G = 32768;  // TMA tiles, 2 boxes x (64 rows x 128 B)
constexpr uint32_t SM_KH = 49152;                         // Khat [64 rows x 128 ch], same swizzled layout
constexpr uint32_t SM_KQ = SM_KH + 16384;                 // [K+ ; Q+] operand  [128 x 128]
constexpr uint32_t SM_T = SM_KQ + 32768;                  // T operand          [64 x 64]
constexpr uint32_t SM_AP = SM_T + 8192;                   // [K*f ; Q*f]        [128 x 128]
constexpr uint32_t SM_APB = SM_AP + 32768;                // K/f                [64 x 128]
constexpr uint32_t SA = 68;                               // row stride (floats) of A and X
constexpr uint32_t SM_AS = SM_AP;                         //   then A  fp32 [64 x 68]
constexpr uint32_t SM_X = SM_AP + 64 * SA * 4;            //   then X = (I+A)^{-1} fp32 [64 x 68]
constexpr uint32_t SM_P = SM_X + 64 * SA * 4;             //   then P bf16 operand [64 x 64]
constexpr uint32_t SM_OFF = SM_AP + 49152;                // off tile operands (32 KB), see below
constexpr uint32_t SM_Y = SM_OFF;                         //   then solve scratch fp32 [32 x 68]
constexpr uint32_t SM_VT = SM_OFF + 16384;                //   then the v tile (TMA, like q/k/g)
constexpr uint32_t SM_OST = SM_OFF + 32768;               // O staging bf16 [64 x 128]
constexpr uint32_t SM_MISC = SM_OST + 16384;
constexpr uint32_t SM_REF = SM_MISC;                      // fp32 [4][128]: Gam_15, Gam_31, Gam_47, Gam_63
constexpr uint32_t SM_CST = SM_REF + 2048;                // fp32 [9][128] per-channel factors
constexpr uint32_t SM_BETA = SM_CST + 4608;               // fp32 [64]
constexpr uint32_t SM_BAR = SM_BETA + 256;                // mbarriers
constexpr uint32_t SM_TPTR = SM_BAR + 128;                // TMEM base address
constexpr uint32_t SM_USED = SM_TPTR + 16;
constexpr uint32_t SMEM_BYTES = SM_USED + 1024;           // + alignment slack
static_assert(SM_P + 8192 <= SM_OFF, "solve buffers overflow their region");
static_assert(SM_KH % 1024 == 0 && SM_VT % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// The off-diagonal tile's A operand spans the whole 32 KB region as 128 rows: rows 32..63
// (K side) and 96..127 (Q side) hold data; its B operand (32 rows) sits in rows 0..31, and
// rows 64..95 are never read back from the accumulator.

// Per-channel factor rows in SM_CST.
enum { CST_M0 = 0, CST_M1, CST_C0, CST_C1, CST_EM0, CST_EG31, CST_E63M1, CST_E63G31, CST_GC, CST_N };

// TMEM column offsets.
constexpr uint32_t TM_AP = 0, TM_OFF = 64, TM_RA = 96, TM_D1 = 128, TM_U = 256, TM_S = 320, TM_SA = 448;
constexpr uint32_t TM_COLS = 512;

// Barriers.
// BAR_OPS .. BAR_UREADY: something the compute threads produce is ready (256 arrivals each): the
// intra-chunk operands, the bf16 state copy (and O of the previous chunk read out), T,
// -(K+ S)^T, U^T.
enum { BAR_TMA = 0, BAR_AP, BAR_M1, BAR_M2, BAR_M34, BAR_V, BAR_OPS, BAR_SREADY, BAR_TREADY, BAR_RREADY, BAR_UREADY,
       BAR_N };

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Offset of the 16-byte chunk (row r, channels 8j..8j+7) in a 64-row TMA tile stored as two
// 64-channel boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_chunk(int r, int j) {
    return (uint32_t)((j >> 3) * 8192 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_chunk(uint8_t *base, uint32_t off, const float (&v)[8]) {
    uint4 w;
    w.x = pack_bf16(v[0], v[1]);
    w.y = pack_bf16(v[2], v[3]);
    w.z = pack_bf16(v[4], v[5]);
    w.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(base + off) = w;
}

// Write 32 consecutive columns k0..k0+31 of row `row` of a K-major bf16 operand with K columns.
__device__ __forceinline__ void st_row32(uint8_t *base, int row, int k0, int K, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(base + kmajor_offset(row, k0 + 8 * q, K)) = w;
    }
}

// 32 floats -> 16 bf16 pairs (element 2i in the low half), optionally negated.
__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&w)[16], float sign) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(sign * v[2 * i], sign * v[2 * i + 1]);
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// One warp: acc[16 x 8] = L[16 x K] * R[K x 8], fp32 row-major shared-memory operands with row
// strides `ls` and `rs` (floats), tf32 inputs and fp32 accumulation (mma.sync m16n8k8).
// acc layout: acc[0] = (g, 2t), acc[1] = (g, 2t+1), acc[2] = (g+8, 2t), acc[3] = (g+8, 2t+1)
// with g = lane / 4, t = lane % 4.
template <int K>
__device__ __forceinline__ void warp_mma_16x8(float (&acc)[4], const float *L, int ls, const float *R, int rs,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint32_t a0 = to_tf32(L[g * ls + k0 + t]), a1 = to_tf32(L[(g + 8) * ls + k0 + t]);
        const uint32_t a2 = to_tf32(L[g * ls + k0 + t + 4]), a3 = to_tf32(L[(g + 8) * ls + k0 + t + 4]);
        const uint32_t b0 = to_tf32(R[(k0 + t) * rs + g]), b1 = to_tf32(R[(k0 + t + 4) * rs + g]);
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Store `scale * acc` (16 x 8 accumulator of warp_mma_16x8) to a row-major fp32 matrix.
__device__ __forceinline__ void warp_store_16x8(float *Out, int os, const float (&acc)[4], float scale, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(Out + g * os + 2 * t) = make_float2(scale * acc[0], scale * acc[1]);
    *reinterpret_cast<float2 *>(Out + (g + 8) * os + 2 * t) = make_float2(scale * acc[2], scale * acc[3]);
}

// T entries of a 16 x 8 accumulator holding -X (rows r0.., columns c0..): T = X Diag(beta),
// written as bf16 pairs into the K-major T operand (64 x 64).
__device__ __forceinline__ void store_t_16x8(uint8_t *Tbase, int r0, int c0, const float (&acc)[4], const float *beta,
                                             int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int cc = c0 + 2 * t;
    const float b0 = -beta[cc], b1 = -beta[cc + 1];
    *reinterpret_cast<uint32_t *>(Tbase + kmajor_offset(r0 + g, cc, 64)) = pack_bf16(acc[0] * b0, acc[1] * b1);
    *reinterpret_cast<uint32_t *>(Tbase + kmajor_offset(r0 + g + 8, cc, 64)) = pack_bf16(acc[2] * b0, acc[3] * b1);
}

// Barrier over the compute threads only (named barrier 1): the issuer warp never joins it.
__device__ __forceinline__ void sync_compute() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

// All compute threads wait on `bar`; true only if every one of them saw the phase complete.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    const uint32_t bad = mbar_wait(bar, parity, kWaitNs) ? 0u : 1u;
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any)
        : "r"(bad), "n"(NT)
        : "memory");
    return any == 0;
}

// Issue `steps` K-steps of one MMA (both operands K-major no-swizzle in shared memory).
__device__ __forceinline__ void issue_mma(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, int K, int steps,
                                          uint32_t idesc, bool accumulate) {
    const uint32_t sbo = (uint32_t)K * 16u;
#pragma unroll 1
    for (int s = 0; s < steps; ++s) {
        const uint64_t a = sdesc(a_smem + 256u * s, 128u, sbo);
        const uint64_t b = sdesc(b_smem + 256u * s, 128u, sbo);
        mma_bf16(d_tmem, a, b, idesc, (accumulate || s > 0) ? 1u : 0u);
    }
}

struct Maps {
    CUtensorMap q, k, g, v;
};

__global__ void __launch_bounds__(NTHREADS, 1)
    kda_prefill_tc_kernel(const __grid_constant__ Maps maps, const RunParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    float *refs = reinterpret_cast<float *>(sm + SM_REF);
    float *cst = reinterpret_cast<float *>(sm + SM_CST);
    float *sbeta = reinterpret_cast<float *>(sm + SM_BETA);
    float *As = reinterpret_cast<float *>(sm + SM_AS);
    float *Xs = reinterpret_cast<float *>(sm + SM_X);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM_BAR);
    uint32_t *tptr = reinterpret_cast<uint32_t *>(sm + SM_TPTR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int h = blockIdx.x % H;
    const int n = blockIdx.x / H;

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
    const int nchunks = (int)((eos - bos + C - 1) / C);

    if (warp == 0) {
        tmem_alloc(tptr, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int b = 0; b < BAR_N; ++b)
            mbar_init(&bars[b], b >= BAR_OPS ? NT : 1);
        fence_mbar_init();
    }
    if (tid == 64) {
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.g);
        prefetch_tensormap(&maps.v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tptr;
    const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter

    // Epilogue mapping: TMEM lane ev (= d_v index), column half eh.
    const int ev = tid & 127, eh = tid >> 7;
    const size_t state_off = ((size_t)n * H + h) * (size_t)D * D;
    const __nv_bfloat16 *bg = static_cast<const __nv_bfloat16 *>(p.beta);
    __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o);

    // Initial state -> TMEM (fp32) and the bf16 S^T operand.
#pragma unroll 1
    for (int cb = 0; cb < 2 && warp < kIssuer; ++cb) {
        const int k0 = 64 * eh + 32 * cb;
        float buf[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            buf[i] = p.init ? __ldcs(p.init + state_off + (size_t)(k0 + i) * D + ev) : 0.f;
        tmem_st32(tmem + tq + TM_S + k0, buf);
        uint32_t w[16];
        pack32(buf, w, 1.f);
        tmem_st16(tmem + tq + TM_SA + k0 / 2, w);
    }
    tmem_st_wait();

    if (tid == 0 && nchunks > 0) {
        mbar_arrive_expect_tx(&bars[BAR_TMA], 3 * 16384);
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sm + SM_Q + 8192 * b, &maps.q, &bars[BAR_TMA], 64 * b, h, (int)bos);
            tma_load_3d(sm + SM_K + 8192 * b, &maps.k, &bars[BAR_TMA], 64 * b, h, (int)bos);
            tma_load_3d(sm + SM_G + 8192 * b, &maps.g, &bars[BAR_TMA], 64 * b, h, (int)bos);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kIssuer) {
        // ---------------------------------------------------------------- issuer warp --------
        if (lane == 0) {
            bool iok = true;
            uint32_t pend = nchunks > 0 ? (1u << BAR_TMA) : 0u;  // operations in flight
            uint32_t tpar = 0;                                    // parity of the TMA phase in flight
            int cc = 0;
#pragma unroll 1
            for (; cc < nchunks; ++cc) {
                const uint32_t par = (uint32_t)(cc & 1);
                const long long row0 = bos + (long long)cc * C;
                if (!(iok = mbar_wait(&bars[BAR_OPS], par, kWaitNs))) break;
                pend = 0;  // the compute side saw this chunk's tiles and every earlier MMA complete
                tc_fence_after();
                issue_mma(tmem + TM_AP, sb + SM_AP, sb + SM_APB, D, D / 16, idesc_bf16(128, 64), false);
                issue_mma(tmem + TM_OFF, sb + SM_OFF, sb + SM_OFF, D, D / 16, idesc_bf16(128, 32), false);
                mma_commit(&bars[BAR_AP]);
                pend |= 1u << BAR_AP;
                if (cc + 1 < nchunks) {  // this chunk's q/k/g tiles are consumed: fetch the next ones
                    const int nr = (int)(row0 + C);
                    mbar_arrive_expect_tx(&bars[BAR_TMA], 3 * 16384);
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(sm + SM_Q + 8192 * b, &maps.q, &bars[BAR_TMA], 64 * b, h, nr);
                        tma_load_3d(sm + SM_K + 8192 * b, &maps.k, &bars[BAR_TMA], 64 * b, h, nr);
                        tma_load_3d(sm + SM_G + 8192 * b, &maps.g, &bars[BAR_TMA], 64 * b, h, nr);
                    }
                    pend |= 1u << BAR_TMA;
                    tpar = (uint32_t)((cc + 1) & 1);
                }
                // MMA1 once the bf16 state copy is in TMEM (and O of the previous chunk is read out)
                if (!(iok = mbar_wait(&bars[BAR_SREADY], par, kWaitNs))) break;
                tc_fence_after();
#pragma unroll 1
                for (int st = 0; st < D / 16; ++st)
                    mma_bf16_tmem_a(tmem + TM_D1, tmem + TM_SA + 8 * st, sdesc(sb + SM_KQ + 256u * st, 128u, 2048u),
                                    idesc_bf16(128, 128), st > 0);
                mma_commit(&bars[BAR_M1]);
                pend |= 1u << BAR_M1;
                // The off-tile operands are consumed: the v tile of this chunk lands in their region.
                if (!(iok = mbar_wait(&bars[BAR_AP], par, kWaitNs))) break;
                pend &= ~(1u << BAR_AP);
                mbar_arrive_expect_tx(&bars[BAR_V], 16384);
                tma_load_3d(sm + SM_VT, &maps.v, &bars[BAR_V], 0, h, (int)row0);
                tma_load_3d(sm + SM_VT + 8192, &maps.v, &bars[BAR_V], 64, h, (int)row0);
                pend |= 1u << BAR_V;
                if (!(iok = mbar_wait(&bars[BAR_V], par, kWaitNs))) break;
                pend &= ~(1u << BAR_V);
                if (!(iok = mbar_wait(&bars[BAR_TREADY], par, kWaitNs))) break;
                // U^T = V^T T^T (V tile as an MN-major A operand) + (-(K+ S)^T from TMEM) T^T; the
                // first half runs while the compute warps move -(K+ S)^T into TMEM.
#pragma unroll 1
                for (int st = 0; st < C / 16; ++st)
                    mma_bf16(tmem + TM_U, sdesc_sw128(sb + SM_VT + 2048u * st, 8192u, 1024u),
                             sdesc(sb + SM_T + 256u * st, 128u, 1024u), idesc_bf16(128, 64) | kIdescAMajorMN, st > 0);
                if (!(iok = mbar_wait(&bars[BAR_RREADY], par, kWaitNs))) break;
                tc_fence_after();
#pragma unroll 1
                for (int st = 0; st < C / 16; ++st)
                    mma_bf16_tmem_a(tmem + TM_U, tmem + TM_RA + 8 * st, sdesc(sb + SM_T + 256u * st, 128u, 1024u),
                                    idesc_bf16(128, 64), 1u);
                mma_commit(&bars[BAR_M2]);
                pend |= 1u << BAR_M2;
                if (!(iok = mbar_wait(&bars[BAR_UREADY], par, kWaitNs))) break;
                tc_fence_after();
#pragma unroll 1
                for (int st = 0; st < C / 16; ++st)
                    mma_bf16_tmem_a(tmem + TM_D1 + 64, tmem + TM_RA + 8 * st, sdesc(sb + SM_P + 256u * st, 128u, 1024u),
                                    idesc_bf16(128, 64), 1u);
#pragma unroll 1
                for (int st = 0; st < C / 16; ++st)
                    mma_bf16_tmem_a(tmem + TM_S, tmem + TM_RA + 8 * st, sdesc_sw128(sb + SM_KH + 2048u * st, 8192u, 1024u),
                                    idesc_bf16(128, 128) | kIdescBMajorMN, 1u);
                mma_commit(&bars[BAR_M34]);
                pend |= 1u << BAR_M34;
            }
            if (!iok) {
                atomicOr(p.err, kErrTimeout);
                // Drain what was issued (bounded), so no MMA or copy is in flight at exit.
                const uint32_t par = (uint32_t)(cc & 1);
                for (int b = 0; b < BAR_N; ++b)
                    if (pend & (1u << b)) (void)mbar_wait(&bars[b], b == BAR_TMA ? tpar : par, kWaitNs);
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------------- compute warps --------
        bool ok = true;
        // Operand mapping: channels 8j..8j+7, rows rlo + 8 * (4 * mh + m) for m = 0..3.
        const int rlo = lane & 7;
        const int j = 4 * (warp & 3) + (lane >> 3);
        const int mh = warp >> 2;
        float gm[4][8];  // Gam of the operand mapping's 4 rows x 8 channels (current chunk)
        // Step 1 of chunk cc: wait for its q/k/g tiles, Gam = cumsum of g into gm, the reference
        // rows and per-channel factors into shared memory, beta into sbeta. Runs for chunk c + 1
        // while the last MMAs of chunk c are in flight. False if the TMA wait ran out.
        auto step1 = [&](int cc) -> bool {
        const long long r0 = bos + (long long)cc * C;
        const int ln = (int)min((long long)C, eos - r0);
        float bet = 0.f;
        if (tid < C && tid < ln) bet = __bfloat162float(bg[(size_t)(r0 + tid) * H + h]);
        if (!wait_all(&bars[BAR_TMA], (uint32_t)(cc & 1))) return false;

        // ---- 1. Gam = cumsum_r g within the chunk, per key channel --------------------------
        // A warp holds 32 consecutive rows of 32 channels: scan over the 8 lanes of a row
        // group with shuffles, then over the 4 row groups in registers; the second row half
        // then adds Gam_31.
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = rlo + 8 * (4 * mh + m);
            const uint4 w = *reinterpret_cast<const uint4 *>(sm + SM_G + tile_chunk(r, j));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) gm[m][i] = r < ln ? ((i & 1) ? bf_hi(ww[i >> 1]) : bf_lo(ww[i >> 1])) : 0.f;
        }
#pragma unroll
        for (int d = 1; d < 8; d <<= 1) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float t = __shfl_up_sync(0xffffffffu, gm[m][i], d, 8);
                    if (rlo >= d) gm[m][i] += t;
                }
            }
        }
        {
            float run[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) run[i] = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float total = __shfl_sync(0xffffffffu, gm[m][i], 7, 8);
                    gm[m][i] += run[i];
                    run[i] += total;
                }
            }
        }
        if (rlo == 7) {  // rows 15 and 31 of the half (half-local sums for the second half)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                refs[(2 * mh) * 128 + 8 * j + i] = gm[1][i];
                refs[(2 * mh + 1) * 128 + 8 * j + i] = gm[3][i];
            }
        }
        if (tid < C) sbeta[tid] = bet;
        sync_compute();
        if (mh) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float g31 = refs[128 + 8 * j + i];
#pragma unroll
                for (int m = 0; m < 4; ++m) gm[m][i] += g31;
            }
        }
        if (tid < 128) {
            const int ch = tid;
            const float G15 = refs[ch], G31 = refs[128 + ch];
            const float G47 = refs[256 + ch] + G31, G63 = refs[384 + ch] + G31;
            cst[CST_M0 * 128 + ch] = G15;
            cst[CST_M1 * 128 + ch] = G47;
            cst[CST_C0 * 128 + ch] = ex2((G31 - G15) * kLog2e);
            cst[CST_C1 * 128 + ch] = ex2((G47 - G31) * kLog2e);
            cst[CST_EM0 * 128 + ch] = ex2(G15 * kLog2e);
            cst[CST_EG31 * 128 + ch] = ex2(G31 * kLog2e);
            cst[CST_E63M1 * 128 + ch] = ex2((G63 - G47) * kLog2e);
            cst[CST_E63G31 * 128 + ch] = ex2((G63 - G31) * kLog2e);
            cst[CST_GC * 128 + ch] = ex2(G63 * kLog2e);
        }
        sync_compute();

        return true;
    };

        // O of a finished chunk (in TMEM columns 192..255) -> staging -> 16-byte coalesced stores.
        auto write_o = [&](long long r0, int ln) {
            float ov[32];
            tmem_ld32(tmem + tq + TM_D1 + 64 + 32 * eh, ov);
            tmem_ld_wait();
            __nv_bfloat16 *ost = reinterpret_cast<__nv_bfloat16 *>(sm + SM_OST);
#pragma unroll
            for (int i = 0; i < 32; ++i) ost[(32 * eh + i) * D + ev] = __float2bfloat16_rn(ov[i]);
            sync_compute();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int idx = tid + NT * q;  // 1024 chunks of 16 bytes: row idx / 16, chunk idx % 16
                const int r = idx >> 4, c16 = idx & 15;
                if (r < ln)
                    *reinterpret_cast<uint4 *>(og + ((size_t)(r0 + r) * H + h) * D + 8 * c16) =
                        *reinterpret_cast<const uint4 *>(sm + SM_OST + r * 256 + 16 * c16);
            }
        };

        int c = 0;
        long long prev_row0 = 0;
        int prev_len = 0;
        if (nchunks > 0) ok = step1(0);
#pragma unroll 1
        for (; ok && c < nchunks; ++c) {
            const uint32_t par = (uint32_t)(c & 1);
            const long long row0 = bos + (long long)c * C;
            const int len = (int)min((long long)C, eos - row0);

        // ---- 2. decay-scaled operands -----------------------------------------------------
        {
            // Per-channel factors of this row half (see the exponent-range note at the top):
            //   rows 0..31 : f = exp(Gam_r - Gam_15); off-tile column factor fi*c0 = exp(Gam_31 - Gam_r)
            //   rows 32..63: f = exp(Gam_r - Gam_47); off-tile row factor    f*c1  = exp(Gam_r - Gam_31)
            float ref[8], fo_c[8], pe[8], khe[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ch = 8 * j + i;
                ref[i] = cst[(mh ? CST_M1 : CST_M0) * 128 + ch];
                fo_c[i] = cst[(mh ? CST_C1 : CST_C0) * 128 + ch];
                pe[i] = cst[(mh ? CST_EG31 : CST_EM0) * 128 + ch];
                khe[i] = cst[(mh ? CST_E63M1 : CST_E63G31) * 128 + ch];
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = rlo + 8 * (4 * mh + m);
                const bool live = r < len;  // rows past the sequence end act as identity tokens
                const uint4 kw = *reinterpret_cast<const uint4 *>(sm + SM_K + tile_chunk(r, j));
                const uint4 qw = *reinterpret_cast<const uint4 *>(sm + SM_Q + tile_chunk(r, j));
                const uint32_t kk[4] = {live ? kw.x : 0u, live ? kw.y : 0u, live ? kw.z : 0u, live ? kw.w : 0u};
                const uint32_t qq[4] = {live ? qw.x : 0u, live ? qw.y : 0u, live ? qw.z : 0u, live ? qw.w : 0u};
                float apk[8], apq[8], apb[8], ofr_k[8], ofr_q[8], kp[8], qp[8], kh[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float kv = (i & 1) ? bf_hi(kk[i >> 1]) : bf_lo(kk[i >> 1]);
                    const float qv = (i & 1) ? bf_hi(qq[i >> 1]) : bf_lo(qq[i >> 1]);
                    // |Gam_r - ref| <= 80 for g in [-5, 0]; the clamp only keeps factors finite
                    // (no 0 * inf) for gates outside that range.
                    const float e = fminf(fmaxf((gm[m][i] - ref[i]) * kLog2e, -126.f), 126.f);
                    const float f = ex2(e), fi = ex2(-e);
                    apk[i] = kv * f;
                    apq[i] = qv * f;
                    apb[i] = kv * fi;
                    // Every other operand is one of these times a per-channel factor <= 1 (so the
                    // product stays in range):
                    if (mh) {                           // rows 32..63
                        ofr_k[i] = apk[i] * fo_c[i];    // K exp(Gam_r - Gam_31): off-tile row
                        ofr_q[i] = apq[i] * fo_c[i];    // Q exp(Gam_r - Gam_31)
                        kp[i] = ofr_k[i] * pe[i];       // K exp(Gam_r)
                        qp[i] = ofr_q[i] * pe[i];       // Q exp(Gam_r)
                        kh[i] = apb[i] * khe[i];        // K exp(Gam_63 - Gam_r)
                    } else {                            // rows 0..31
                        ofr_k[i] = apb[i] * fo_c[i];    // K exp(Gam_31 - Gam_r): off-tile column
                        ofr_q[i] = 0.f;
                        kp[i] = apk[i] * pe[i];         // K exp(Gam_r)
                        qp[i] = apq[i] * pe[i];         // Q exp(Gam_r)
                        kh[i] = ofr_k[i] * khe[i];      // K exp(Gam_63 - Gam_r)
                    }
                }
                st_chunk(sm, SM_AP + kmajor_offset(r, 8 * j, D), apk);
                st_chunk(sm, SM_AP + kmajor_offset(64 + r, 8 * j, D), apq);
                st_chunk(sm, SM_APB + kmajor_offset(r, 8 * j, D), apb);
                st_chunk(sm, SM_OFF + kmajor_offset(r, 8 * j, D), ofr_k);
                if (mh) st_chunk(sm, SM_OFF + kmajor_offset(64 + r, 8 * j, D), ofr_q);
                st_chunk(sm, SM_KQ + kmajor_offset(r, 8 * j, D), kp);
                st_chunk(sm, SM_KQ + kmajor_offset(64 + r, 8 * j, D), qp);
                st_chunk(sm, SM_KH + tile_chunk(r, j), kh);  // row-major: MMA4 reads it MN-major
            }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[BAR_OPS]);

        // ---- 2b. while the intra-chunk tiles run: O of the previous chunk, then the bf16 copy
        //          of the state for MMA1 (the initial state's copy was made before the loop).
        if (c > 0) {
            write_o(prev_row0, prev_len);
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                const int k0 = 64 * eh + 32 * cb;
                float sv[32];
                tmem_ld32(tmem + tq + TM_S + k0, sv);
                tmem_ld_wait();
                uint32_t w[16];
                pack32(sv, w, 1.f);
                tmem_st16(tmem + tq + TM_SA + k0 / 2, w);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars[BAR_SREADY]);

        // ---- 3. the state decay runs in the shadow of the intra-chunk tiles -----------------
        // S <- S Diag(gam_last): the state in TMEM is next read by MMA4 of this chunk.
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            const int k0 = 64 * eh + 32 * cb;
            float sv[32];
            tmem_ld32(tmem + tq + TM_S + k0, sv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[i] *= cst[CST_GC * 128 + k0 + i];
            tmem_st32(tmem + tq + TM_S + k0, sv);
        }
        tmem_st_wait();

        // ---- 4. A (fp32, for the solve) and P (bf16 operand) out of TMEM -------------------
        if (!(ok = wait_all(&bars[BAR_AP], par))) break;
        tc_fence_after();
        {
            const int L = 32 * (warp & 3) + lane;
            const int i = L & 63;
            const bool pside = L >= 64;
            const int jh = warp >> 2;
            float vals[32];
            if (jh == 0) {
                tmem_ld32(tmem + tq + ((i < 32) ? TM_AP : TM_OFF), vals);
                tmem_ld_wait();
            } else if (i >= 32) {
                tmem_ld32(tmem + tq + TM_AP + 32, vals);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) vals[q] = 0.f;
            }
            const int j0 = 32 * jh;
            if (!pside) {
                const float b = sbeta[i];
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    float4 w;
                    w.x = (j0 + q + 0 < i) ? vals[q + 0] * b : 0.f;
                    w.y = (j0 + q + 1 < i) ? vals[q + 1] * b : 0.f;
                    w.z = (j0 + q + 2 < i) ? vals[q + 2] * b : 0.f;
                    w.w = (j0 + q + 3 < i) ? vals[q + 3] * b : 0.f;
                    *reinterpret_cast<float4 *>(As + i * SA + j0 + q) = w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) vals[q] = (j0 + q <= i) ? vals[q] : 0.f;
                st_row32(sm + SM_P, i, j0, C, vals);
            }
        }
        sync_compute();

        // ---- 5. X = (I + A)^{-1}, written to T = X Diag(beta) as it completes ------------------
        // (a) warp b < 4 inverts the 16 x 16 diagonal block b by doubling: four 4 x 4 blocks in
        //     closed form, then 4 -> 8 -> 16 merges X21 = -X22 (A21 X11); warps 4..7 zero the
        //     strictly-upper blocks of T and the two upper blocks of X the merges read.
        if (warp < 4) {
            const int B0 = 16 * warp;
            float *Yw = reinterpret_cast<float *>(sm + SM_Y) + warp * (16 * 17);
#pragma unroll
            for (int q = 0; q < 3; ++q) {  // zero the upper 4 x 4 blocks of the diagonal block
                const int e = lane + 32 * q;   // 96 entries: 6 blocks x 16
                const int blk = e >> 4, rr = (e >> 2) & 3, cc = e & 3;
                const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                Xs[(B0 + 4 * bi + rr) * SA + B0 + 4 * bj + cc] = 0.f;
            }
            if (lane < 4) {  // 4 x 4 unit lower-triangular inverse in closed form
                const int o = B0 + 4 * lane;
                const float a10 = As[(o + 1) * SA + o], a20 = As[(o + 2) * SA + o], a21 = As[(o + 2) * SA + o + 1];
                const float a30 = As[(o + 3) * SA + o], a31 = As[(o + 3) * SA + o + 1], a32 = As[(o + 3) * SA + o + 2];
                const float x10 = -a10, x21 = -a21, x32 = -a32;
                const float x20 = -fmaf(a21, x10, a20);
                const float x31 = -fmaf(a32, x21, a31);
                const float x30 = -fmaf(a32, x20, fmaf(a31, x10, a30));
                float *X0 = Xs + o * SA + o;
                X0[0] = 1.f;      X0[1] = 0.f;      X0[2] = 0.f;      X0[3] = 0.f;
                X0[SA] = x10;     X0[SA + 1] = 1.f; X0[SA + 2] = 0.f; X0[SA + 3] = 0.f;
                X0[2 * SA] = x20; X0[2 * SA + 1] = x21; X0[2 * SA + 2] = 1.f; X0[2 * SA + 3] = 0.f;
                X0[3 * SA] = x30; X0[3 * SA + 1] = x31; X0[3 * SA + 2] = x32; X0[3 * SA + 3] = 1.f;
            }
            __syncwarp();
            {  // 4 -> 8: lane = (half q, row r, column c) of the two 4 x 4 blocks X21
                const int q = lane >> 4, r = (lane >> 2) & 3, cc = lane & 3;
                const int o = B0 + 8 * q;
                float y = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) y = fmaf(As[(o + 4 + r) * SA + o + m], Xs[(o + m) * SA + o + cc], y);
                Yw[(4 * q + r) * 17 + cc] = y;
                __syncwarp();
                float x = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) x = fmaf(Xs[(o + 4 + r) * SA + o + 4 + m], Yw[(4 * q + m) * 17 + cc], x);
                Xs[(o + 4 + r) * SA + o + cc] = -x;
            }
            __syncwarp();
            {  // 8 -> 16: X21 (8 x 8), two entries per lane
                const int r = lane >> 2, c0 = (lane & 3) * 2;
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float am = As[(B0 + 8 + r) * SA + B0 + m];
                    y0 = fmaf(am, Xs[(B0 + m) * SA + B0 + c0], y0);
                    y1 = fmaf(am, Xs[(B0 + m) * SA + B0 + c0 + 1], y1);
                }
                Yw[r * 17 + c0] = y0;
                Yw[r * 17 + c0 + 1] = y1;
                __syncwarp();
                float x0 = 0.f, x1 = 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float xm = Xs[(B0 + 8 + r) * SA + B0 + 8 + m];
                    x0 = fmaf(xm, Yw[m * 17 + c0], x0);
                    x1 = fmaf(xm, Yw[m * 17 + c0 + 1], x1);
                }
                Xs[(B0 + 8 + r) * SA + B0 + c0] = -x0;
                Xs[(B0 + 8 + r) * SA + B0 + c0 + 1] = -x1;
            }
            __syncwarp();
            {  // T of the diagonal block: one 16-byte chunk (row r, 8 columns) per lane
                const int r = lane >> 1, h8 = (lane & 1) * 8;
                float tv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) tv[q] = Xs[(B0 + r) * SA + B0 + h8 + q] * sbeta[B0 + h8 + q];
                st_chunk(sm, SM_T + kmajor_offset(B0 + r, B0 + h8, C), tv);
            }
        } else {
            const int z = tid - 128;  // 0..127
            // X rows 0..15 cols 16..31 and rows 32..47 cols 48..63 (read by the 32 -> 64 merge)
            const int blk = z >> 6, rr = (z & 63) >> 2, cq = (z & 3) * 4;
            *reinterpret_cast<float4 *>(Xs + (32 * blk + rr) * SA + 32 * blk + 16 + cq) = make_float4(0.f, 0.f, 0.f, 0.f);
            // T: the six strictly-upper 16 x 16 blocks (192 chunks of 16 bytes)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int e = z + 128 * q;
                if (e < 192) {
                    const int bi = e >> 5, r2 = (e & 31) >> 1, hf = e & 1;
                    const int I = bi < 3 ? 0 : (bi < 5 ? 1 : 2);
                    const int J = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
                    *reinterpret_cast<uint4 *>(sm + SM_T + kmajor_offset(16 * I + r2, 16 * J + 8 * hf, C)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        sync_compute();
        // (b) 16 -> 32: warp (p, nt) < 4 computes column tile nt of X_{2p+1,2p} (tf32 mma)
        if (warp < 4) {
            const int pp = warp >> 1, nt = warp & 1;
            const int I = 2 * pp + 1, J = 2 * pp;
            float *Yb = reinterpret_cast<float *>(sm + SM_Y + 4352) + 16 * pp * SA;
            float acc[4];
            warp_mma_16x8<16>(acc, As + 16 * I * SA + 16 * J, SA, Xs + 16 * J * SA + 16 * J + 8 * nt, SA, lane);
            warp_store_16x8(Yb + 8 * nt, SA, acc, 1.f, lane);
            __syncwarp();
            warp_mma_16x8<16>(acc, Xs + 16 * I * SA + 16 * I, SA, Yb + 8 * nt, SA, lane);
            warp_store_16x8(Xs + 16 * I * SA + 16 * J + 8 * nt, SA, acc, -1.f, lane);
            store_t_16x8(sm + SM_T, 16 * I, 16 * J + 8 * nt, acc, sbeta, lane);
        }
        sync_compute();
        // (c) 32 -> 64: X_BA = -X_BB A_BA X_AA with 32 x 32 blocks; warp w owns one 16 x 8 tile.
        {
            const int mt = warp >> 2, nt = warp & 3;
            float *Y = reinterpret_cast<float *>(sm + SM_Y + 4352);
            float acc[4];
            warp_mma_16x8<32>(acc, As + (32 + 16 * mt) * SA, SA, Xs + 8 * nt, SA, lane);
            warp_store_16x8(Y + 16 * mt * SA + 8 * nt, SA, acc, 1.f, lane);
            sync_compute();
            warp_mma_16x8<32>(acc, Xs + (32 + 16 * mt) * SA + 32, SA, Y + 8 * nt, SA, lane);
            store_t_16x8(sm + SM_T, 32 + 16 * mt, 8 * nt, acc, sbeta, lane);
        }

        // ---- 6. U = T V - T (K+ S): -(K+ S)^T goes to TMEM as MMA2's second A operand ----------
        fence_async_smem();  // the T stores of the solve
        mbar_arrive(&bars[BAR_TREADY]);
        if (!(ok = wait_all(&bars[BAR_M1], par))) break;
        tc_fence_after();
        {
            float ks[32];
            tmem_ld32(tmem + tq + TM_D1 + 32 * eh, ks);
            tmem_ld_wait();
            uint32_t w[16];
            pack32(ks, w, -1.f);
            tmem_st16(tmem + tq + TM_RA + 16 * eh, w);
            tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars[BAR_RREADY]);

        if (!(ok = wait_all(&bars[BAR_M2], par))) break;
        tc_fence_after();
        {
            float u[32];
            tmem_ld32(tmem + tq + TM_U + 32 * eh, u);
            tmem_ld_wait();
            uint32_t w[16];
            pack32(u, w, 1.f);
            tmem_st16(tmem + tq + TM_RA + 16 * eh, w);  // U^T replaces -(K+ S)^T (MMA2 has finished)
            tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars[BAR_UREADY]);

        if (c + 1 < nchunks && !(ok = step1(c + 1))) break;
        if (!(ok = wait_all(&bars[BAR_M34], par))) break;
        tc_fence_after();

        prev_row0 = row0;
        prev_len = len;
        }

        if (ok && nchunks > 0) write_o(prev_row0, prev_len);  // O of the last chunk
        if (ok) {
            if (p.fin) {
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    const int k0 = 64 * eh + 32 * cb;
                    float sv[32];
                    tmem_ld32(tmem + tq + TM_S + k0, sv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) __stcs(p.fin + state_off + (size_t)(k0 + i) * D + ev, sv[i]);
                }
            }
        } else if (tid == 0) {
            atomicOr(p.err, kErrTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool encode_map(CUtensorMap *map, const void *base, long long rows, int H) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p) {
    if (dtype != KDA_BF16 || dk != D || dv != D) return false;
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    if (rows <= 0 || rows > 0x7fffffffLL - C) return false;
    return tensor_map_encoder() != nullptr;
}

cudaError_t launch_tc_prefill(const RunParams &p, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(kda_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    Maps maps;
    if (!encode_map(&maps.q, p.q, rows, p.H) || !encode_map(&maps.k, p.k, rows, p.H) ||
        !encode_map(&maps.g, p.g, rows, p.H) || !encode_map(&maps.v, p.v, rows, p.H))
        return cudaErrorInvalidValue;
    kda_prefill_tc_kernel<<<(unsigned)(p.n_seqs * p.H), NTHREADS, SMEM_BYTES, s>>>(maps, p);
    return cudaGetLastError();
}

}  // namespace kda
