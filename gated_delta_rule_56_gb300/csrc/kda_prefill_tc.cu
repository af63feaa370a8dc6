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
// Layout of the work: one CTA per (sequence, head); chunks run in order, in two overlapped
// streams of work carried by different warps:
//   prep warps 0..7    the state-independent work of a chunk: Gam (cumsum of g, thread = 4
//                      consecutive rows x 8 channels), the decay-scaled operands, and the block
//                      merges of T = (I + A)^{-1} Diag(beta). While the A/P MMAs of chunk c run
//                      they already compute Gam of chunk c + 1.
//   state warps 8..11  thread = TMEM lane = value column: the bf16 state copy fused with the
//                      decay S <- S Diag(gam_last), A and P out of TMEM and the 16 x 16 diagonal
//                      blocks of the inverse, -(K+ S)^T and U^T as bf16 A operands in TMEM, and O
//                      of chunk c - 1 out while the prep warps merge the inverse of chunk c (read
//                      from TMEM in the MMA-fragment layout, stored transposed by stmatrix into the
//                      TMA tile layout in shared memory, one TMA tensor store per 64 channels).
//   issuer warp 12     the whole warp walks the chunks and one elected lane issues every MMA and
//                      TMA copy, in the order the work becomes ready; mbarriers carry each
//                      hand-off between the three groups.
//   TMA: g (fetched by the prep warps), q/k of the next chunk as soon as the current ones are
//        read, v once MMA2 has read the last; every tile 64 rows x 128 channels, 128-byte swizzle.
//   TMEM (512 columns): [0,64) diagonal A|P tile, [64,96) off-diagonal tile, [96,128) the
//        bf16 A operand -(K+ S)^T then U^T, [128,192) K+ S then U, [192,256) and [256,320) the
//        Q+ S -> O accumulators of even and odd chunks (O of chunk c is read out while chunk
//        c + 1 runs), [320,448) the fp32 state S^T (lanes = d_v), [448,512) its bf16 copy.
//   MMAs (kind::f16, bf16 operands, fp32 accumulate; "tmem" = A read from TMEM; shared-memory
//   operands in the 128-byte-swizzled layout):
//        diag  [K*f ; Q*f] x [K/f]^T              M = 128, N = 64, K = 128
//        off   [K*e ; Q*e] x [K*e']^T             M = 64,  N = 32, K = 128
//        MMA1  S^T (tmem) x [K+ ; Q+]^T           M = 128, two N = 64 halves, K = 128
//        MMA2  V^T x T^T  (V tile, MN-major)      N = 64,  K = 64    -> then += -(K+ S)^T (tmem) x T^T = U^T
//                                                                      (into the columns of K+ S, once read)
//        MMA3  U^T (tmem) x P^T  (onto (Q+ S)^T)  N = 64,  K = 64    -> O^T
//        MMA4  U^T (tmem) x Khat  (MN-major B)    N = 128, K = 64    -> S^T
//   MMA1 starts as soon as the operands and the state copy exist. Once it has read [K+ ; Q+], that
//   region stages O of the previous chunk for its TMA store; the prep warps build the next chunk's
//   [K+ ; Q+] there after the store has read it (KQFREE).
//   The 64 x 64 triangular inverse: 16 x 16 diagonal blocks by doubling on CUDA cores, then the
//   16->32 and 32->64 block merges as tf32 warp-level MMAs.
// Every mbarrier wait is bounded; on time-out the CTA records kErrTimeout, drains what it
// issued (again bounded), frees its TMEM and exits.
//
// Instances (template flags, chosen at launch): gate logits (g = -bound * sigmoid(x) formed as
// g is read), q/k L2 normalisation (row sums of squares before the operands are built) and the
// output gate (O scaled by sigmoid(z) as it is staged). The same kernel also runs the passes of
// the split long-sequence prefill (kda_segmented.cu): v taken as zero, the identity as the start
// state, a cap on the chunks run, and a per-(sequence, head) skip list.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;                     // chunk length
constexpr int D = 128;                    // d_k == d_v
constexpr int NP = 256;                   // prep threads (warps 0..7)
constexpr int NS = 128;                   // state threads (warps 8..11), thread = TMEM lane = d_v index
constexpr int kStateWarp0 = NP / 32;
constexpr int kIssuer = (NP + NS) / 32;   // warp 12 issues every MMA and TMA copy
constexpr int NTHREADS = NP + NS + 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait

// Shared memory map (bytes from a 1024-byte aligned base). The decay-scaled operands (and the TMA
// tiles) use the 128-byte-swizzled K-major layout: in an R-row operand, the 16-byte chunk (row r,
// channels 8j..8j+7) sits at sw_chunk(r, j, R) (rows of 128 B = 64 channels, 8-row atoms of 1 KB,
// the second 64 channels R * 128 bytes further on), so the 8 chunks of one row are bank-free.
constexpr uint32_t SM_Q = 0, SM_K = 16384, SM_G = 32768;  // TMA tiles, 2 boxes x (64 rows x 128 B)
constexpr uint32_t SM_KH = 49152;                         // Khat, two buffers of [64 rows x 128 ch] (TMA layout)
constexpr uint32_t SM_KQ = SM_KH + 32768;                 // [K+ ; Q+] operand  [128 rows x 128]
constexpr uint32_t SM_T = SM_KQ + 32768;                  // T operand          [64 x 64]
constexpr uint32_t SM_P = SM_T + 8192;                    // P operand          [64 x 64]
constexpr uint32_t SM_AP = SM_P + 8192;                   // [K*f ; Q*f]        [128 rows x 128]
constexpr uint32_t SM_APB = SM_AP + 32768;                // K/f                [64 rows x 128]
constexpr uint32_t SA = 68;                               // row stride (floats) of A and X
constexpr uint32_t SM_AS = SM_AP;                         //   then A  fp32 [64 x 68]
constexpr uint32_t SM_X = SM_AP + 64 * SA * 4;            //   then X = (I+A)^{-1} fp32 [64 x 68]
constexpr uint32_t SM_OFF = SM_AP + 49152;                // off tile: A operand [64 rows x 128] ...
constexpr uint32_t SM_OFFB = SM_OFF + 16384;              //   ... and B operand [32 rows x 128]
constexpr uint32_t SM_Y = SM_OFF;                         //   then solve scratch fp32
constexpr uint32_t SM_VT = SM_OFF + 24576;                // v tile (TMA, like q/k/g)
constexpr uint32_t SM_MISC = SM_VT + 16384;
constexpr uint32_t SM_WT = SM_MISC;                       // fp32 [4][128]: sums of g over each 16-row block
constexpr uint32_t SM_CST = SM_WT + 2048;                // fp32 [8][128] per-channel factors
constexpr uint32_t SM_GC = SM_CST + 4096;                 // fp32 [3][128] gam_last, by chunk index mod 3
constexpr uint32_t SM_BETA = SM_GC + 1536;                // fp32 [2][64] beta, by chunk parity
constexpr uint32_t SM_BAR = SM_BETA + 512;                // mbarriers
constexpr uint32_t SM_TPTR = SM_BAR + 256;                // TMEM base address
constexpr uint32_t SM_NRM = SM_TPTR + 16;                 // fp32 [3 chunks][k, q][64]: row sums of squares
constexpr uint32_t SM_USED = SM_NRM + 1536;
constexpr uint32_t SMEM_BYTES = SM_USED + 1024;           // + alignment slack
static_assert(SM_X + 64 * SA * 4 <= SM_OFF, "solve buffers overflow their region");
constexpr uint32_t SM_YC = SM_Y + 4352 + 32 * SA * 4;  //   and the 32 -> 64 merge's product A_BA X_AA
static_assert(SM_YC + 32 * SA * 4 <= SM_VT, "solve scratch overflows its region");
static_assert(SM_KH % 1024 == 0 && SM_KQ % 1024 == 0 && SM_AP % 1024 == 0 && SM_APB % 1024 == 0 &&
                  SM_OFF % 1024 == 0 && SM_OFFB % 1024 == 0 && SM_VT % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Per-channel factor rows in SM_CST.
enum { CST_C0 = 0, CST_C1, CST_EM0, CST_EG31, CST_E63M1, CST_E63G31, CST_N };
static_assert(CST_N * 512 <= 4096, "factor rows overflow SM_CST");

// TMEM column offsets.
constexpr uint32_t TM_AP = 0, TM_OFF = 64, TM_RA = 96, TM_D1 = 128, TM_S = 320, TM_SA = 448;
// O (Q+ S, then += P U) of chunk c in one of two slots by chunk parity, so that MMA1 of chunk c + 1
// can run before O of chunk c has been read out.
constexpr uint32_t TM_O0 = TM_D1 + 64, TM_O1 = 256;
__device__ __forceinline__ uint32_t o_slot(int c) { return (c & 1) ? TM_O1 : TM_O0; }
constexpr uint32_t TM_COLS = 512;

// Barriers. Up to BAR_DRAIN: TMA copies and MMA commits (one arrival; BAR_M1 = the K+ half of
// MMA1, BAR_M1Q = all of MMA1). BAR_OPS, BAR_TREADY, BAR_S1D0/1: the prep warps have built the
// intra-chunk operands / written T / finished step 1 of an even / odd chunk (gam_last and beta in
// place) (NP arrivals). BAR_SREADY .. BAR_KQFREE: the state warps have made the bf16 state copy /
// -(K+ S)^T / U^T / A, P and the diagonal blocks of the inverse / released the [K+ ; Q+] region
// (MMA1 has read it and the O store of the previous chunk has read its staging) (NS arrivals).
enum {
    BAR_G = 0, BAR_QK, BAR_V, BAR_AP, BAR_M1, BAR_M1Q, BAR_M2, BAR_M34, BAR_DRAIN,
    BAR_OPS, BAR_TREADY, BAR_S1D0, BAR_S1D1,
    BAR_SREADY, BAR_RREADY, BAR_UREADY, BAR_EPIDONE, BAR_KQFREE,
    BAR_N
};
static_assert(BAR_N * 8 <= 256, "barrier region");

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight consecutive floats from 16-byte aligned shared memory.
__device__ __forceinline__ void lds8(float (&d)[8], const float *src) {
    const float4 a = *reinterpret_cast<const float4 *>(src), b = *reinterpret_cast<const float4 *>(src + 4);
    d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w; d[4] = b.x; d[5] = b.y; d[6] = b.z; d[7] = b.w;
}
// Two fp32 products in one instruction (each rounded to nearest, as two separate products).
__device__ __forceinline__ void mul2(float &a, float &b, float x, float y) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(a)),
          "l"(((uint64_t)__float_as_uint(y) << 32) | __float_as_uint(x)));
    a = __uint_as_float((uint32_t)r);
    b = __uint_as_float((uint32_t)(r >> 32));
}

// 16 TMEM lanes x 64 fp32 columns in the MMA-fragment layout (tcgen05.ld 16x256b, 8 repetitions):
// register 4k + 0/1 = (lane g, columns 8k + 2t, + 1), 4k + 2/3 = (lane g + 8, the same columns),
// with g = thread / 4 and t = thread % 4 of the warp; taddr's lane field selects the 16 lanes.
__device__ __forceinline__ void tmem_ld_frag64(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// The inverse of stmatrix_x4_trans: four 8 x 8 bf16 matrices read transposed into fragments.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t saddr, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(saddr)
                 : "memory");
}

// Four 8 x 8 bf16 matrices, each stored transposed: lane 8i + j gives the address of row j of
// the transpose of matrix i; each thread's register i holds its fragment of matrix i.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a),
                 "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Offset of the 16-byte chunk (row r, channels 8j..8j+7) in an R-row operand in the 128-byte
// swizzled K-major layout (a 64-row TMA tile of two 64-channel boxes is the R = 64 case).
__device__ __forceinline__ uint32_t sw_chunk(int r, int j, int R) {
    return (uint32_t)((j >> 3) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 + (((j & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t tile_chunk(int r, int j) { return sw_chunk(r, j, 64); }

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
template <int K, bool INIT = true>
__device__ __forceinline__ void warp_mma_16x8(float (&acc)[4], const float *L, int ls, const float *R, int rs,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    if (INIT) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
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

// Barrier over one warp group only (named barrier ID with N threads).
template <int ID, int N>
__device__ __forceinline__ void group_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}

// Every thread of a warp group waits on `bar` (and then on `bar2`, if given: two waits share one
// group barrier); true only if all of them saw the phases complete, so the group leaves its loop
// together when a wait runs out.
template <int ID, int N>
__device__ __forceinline__ bool group_wait(uint64_t *bar, uint32_t parity, uint64_t *bar2 = nullptr,
                                           uint32_t parity2 = 0) {
    uint32_t bad = mbar_wait(bar, parity, kWaitNs) ? 0u : 1u;
    if (!bad && bar2) bad = mbar_wait(bar2, parity2, kWaitNs) ? 0u : 1u;
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any)
        : "r"(bad), "n"(ID), "n"(N)
        : "memory");
    return any == 0;
}

__device__ __forceinline__ void prep_sync() { group_sync<1, NP>(); }
__device__ __forceinline__ bool prep_wait(uint64_t *bar, uint32_t parity, uint64_t *bar2 = nullptr,
                                          uint32_t parity2 = 0) {
    return group_wait<1, NP>(bar, parity, bar2, parity2);
}
__device__ __forceinline__ bool state_wait(uint64_t *bar, uint32_t parity) { return group_wait<2, NS>(bar, parity); }
__device__ __forceinline__ void state_sync() { group_sync<2, NS>(); }

// Decay-scaled bf16 operands of one row half (MH = 0: rows 0..31, MH = 1: rows 32..63) for a
// thread's 4 rows r0..r0+3 x 8 channels 8j..8j+7; gm holds Gam_r - Gam_ref of those entries
// (ref = row 15 for MH = 0, row 47 for MH = 1; summed within the 16-row blocks, so no large
// cumulative values cancel). With the L2
// normalisation (NORM) the operands of the A/P tiles are built from the raw q/k rows, which are
// exact bf16 values, and the A/P read-out applies the inverse norms to the fp32 products: a
// normalised row rounded to bf16 before the product would put an absolute error of about
// 2^-9 / sqrt(d_k) into q.k, a large relative error where q.k is small. Only the operands of the
// products with the state (K+, Q+, Khat) carry the norm.
// Per-channel factors (see the exponent-range note at the top):
//   rows 0..31 : f = exp(Gam_r - Gam_15); off-tile column factor fi*c0 = exp(Gam_31 - Gam_r)
//   rows 32..63: f = exp(Gam_r - Gam_47); off-tile row factor    f*c1  = exp(Gam_r - Gam_31)
// Every other operand is one of K f, Q f, K / f times a per-channel factor <= 1, so each
// product stays in range. Rows past the sequence end (r >= len) act as identity tokens.
// Row sums of squares of k and q for the L2 normalisation, one buffer per chunk index mod 3:
// step 1 of chunk c adds into buffer c % 3 (and zeroes buffer (c + 1) % 3, last read by the
// operands of chunk c - 2), then replaces each sum s by 1 / sqrt(s + 1e-6); the operands and the
// A/P read-out of chunk c read it after step 1's closing barrier.
// The thread's 4 rows x 8 channels of q and k come from global memory (the same lines the TMA
// fetches for the operands later). Each thread sums its 8 channels per row; the 8 lanes of a row
// group reduce the 8 sums (4 k rows, 4 q rows) by halving exchanges, lane i ending with sum i,
// and add it to the row's entry, which the warp holding the other channel half adds to as well.
struct QKRows {
    uint4 k[4], q[4];
};

__device__ __forceinline__ void load_qk_rows(QKRows &x, const __nv_bfloat16 *qg, const __nv_bfloat16 *kg,
                                             long long row0, int ln, int H, int h, int r0, int j, int dg) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const bool live = r0 + m < ln && 8 * j < dg;
        const size_t e = ((size_t)(row0 + r0 + m) * H + h) * dg + 8 * j;
        x.k[m] = live ? __ldg(reinterpret_cast<const uint4 *>(kg + e)) : make_uint4(0u, 0u, 0u, 0u);
        x.q[m] = live ? __ldg(reinterpret_cast<const uint4 *>(qg + e)) : make_uint4(0u, 0u, 0u, 0u);
    }
}

__device__ __forceinline__ void add_row_square_sums(float *nrm, const QKRows &x, int r0, int lane) {
    float v[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t kk[4] = {x.k[m].x, x.k[m].y, x.k[m].z, x.k[m].w};
        const uint32_t qq[4] = {x.q[m].x, x.q[m].y, x.q[m].z, x.q[m].w};
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float kv = (i & 1) ? bf_hi(kk[i >> 1]) : bf_lo(kk[i >> 1]);
            const float qv = (i & 1) ? bf_hi(qq[i >> 1]) : bf_lo(qq[i >> 1]);
            sk = fmaf(kv, kv, sk);
            sq = fmaf(qv, qv, sq);
        }
        v[m] = sk;
        v[4 + m] = sq;
    }
    const int i = lane & 7;
    float w4[4], w2[2];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const bool hi = (i & 4) != 0;
        w4[t] = (hi ? v[4 + t] : v[t]) + __shfl_xor_sync(0xffffffffu, hi ? v[t] : v[4 + t], 4);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const bool hi = (i & 2) != 0;
        w2[t] = (hi ? w4[2 + t] : w4[t]) + __shfl_xor_sync(0xffffffffu, hi ? w4[t] : w4[2 + t], 2);
    }
    const bool hi = (i & 1) != 0;
    const float tot = (hi ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, hi ? w2[0] : w2[1], 1);
    atomicAdd(nrm + (i >> 2) * 64 + r0 + (i & 3), tot);
}

// 1 / sqrt(sum x^2 + 1e-6) of row r of k (kq = 0) or q (kq = 1) from a completed buffer (step 1
// turns the sums into these values once, between its two barriers).
__device__ __forceinline__ float row_inv_norm(const float *nrm, int kq, int r) { return nrm[kq * 64 + r]; }

template <int MH, bool NORM, int ROWS>
__device__ __forceinline__ void build_operands(uint8_t *sm, const float (&gm)[4][8], const float *cst, int r0,
                                               int j, int len, uint32_t khb, const float *nrm) {
    float fo_c[8], pe[8], khe[8];
    lds8(fo_c, cst + (MH ? CST_C1 : CST_C0) * 128 + 8 * j);
    lds8(pe, cst + (MH ? CST_EG31 : CST_EM0) * 128 + 8 * j);
    lds8(khe, cst + (MH ? CST_E63M1 : CST_E63G31) * 128 + 8 * j);
    // ROWS rows per loop iteration (fully unrolled, the body's instructions cost more to fetch than
    // the loop saves). Two: each element's Gam is one of two registers; one: a 4-way select, but
    // 4.6 KB less code, which is faster when every SM of the GPU runs a CTA (see the launch).
#pragma unroll ROWS
    for (int m = 0; m < 4; ++m) {
        const int r = r0 + m;
        const bool live = r < len;
        float gr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) gr[i] = m == 0 ? gm[0][i] : (m == 1 ? gm[1][i] : (m == 2 ? gm[2][i] : gm[3][i]));
        const uint4 kw = *reinterpret_cast<const uint4 *>(sm + SM_K + tile_chunk(r, j));
        const uint4 qw = *reinterpret_cast<const uint4 *>(sm + SM_Q + tile_chunk(r, j));
        const uint32_t kk[4] = {live ? kw.x : 0u, live ? kw.y : 0u, live ? kw.z : 0u, live ? kw.w : 0u};
        const uint32_t qq[4] = {live ? qw.x : 0u, live ? qw.y : 0u, live ? qw.z : 0u, live ? qw.w : 0u};
        const float nk = NORM ? row_inv_norm(nrm, 0, r) : 1.f, nq = NORM ? row_inv_norm(nrm, 1, r) : 1.f;
        float apk[8], apq[8], apb[8], ofr_k[8], ofr_q[8], kp[8], qp[8], kh[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {  // channel pairs, two products per instruction
            const float k0 = bf_lo(kk[i >> 1]), k1 = bf_hi(kk[i >> 1]);
            const float q0 = bf_lo(qq[i >> 1]), q1 = bf_hi(qq[i >> 1]);
            // |Gam_r - ref| <= 80 for g in [-5, 0]; the clamp only keeps factors finite (no 0 * inf)
            // for gates outside that range.
            float e0 = gr[i], e1 = gr[i + 1];  // Gam_r - Gam_ref
            mul2(e0, e1, kLog2e, kLog2e);
            e0 = fminf(fmaxf(e0, -126.f), 126.f);
            e1 = fminf(fmaxf(e1, -126.f), 126.f);
            const float f0 = ex2(e0), f1 = ex2(e1), fi0 = ex2(-e0), fi1 = ex2(-e1);
            apk[i] = k0; apk[i + 1] = k1; mul2(apk[i], apk[i + 1], f0, f1);
            apq[i] = q0; apq[i + 1] = q1; mul2(apq[i], apq[i + 1], f0, f1);
            apb[i] = k0; apb[i + 1] = k1; mul2(apb[i], apb[i + 1], fi0, fi1);
            if (MH) {
                ofr_k[i] = apk[i]; ofr_k[i + 1] = apk[i + 1]; mul2(ofr_k[i], ofr_k[i + 1], fo_c[i], fo_c[i + 1]);
                ofr_q[i] = apq[i]; ofr_q[i + 1] = apq[i + 1]; mul2(ofr_q[i], ofr_q[i + 1], fo_c[i], fo_c[i + 1]);
                kp[i] = ofr_k[i]; kp[i + 1] = ofr_k[i + 1]; mul2(kp[i], kp[i + 1], pe[i], pe[i + 1]);
                qp[i] = ofr_q[i]; qp[i + 1] = ofr_q[i + 1]; mul2(qp[i], qp[i + 1], pe[i], pe[i + 1]);
                kh[i] = apb[i]; kh[i + 1] = apb[i + 1]; mul2(kh[i], kh[i + 1], khe[i], khe[i + 1]);
            } else {
                ofr_k[i] = apb[i]; ofr_k[i + 1] = apb[i + 1]; mul2(ofr_k[i], ofr_k[i + 1], fo_c[i], fo_c[i + 1]);
                kp[i] = apk[i]; kp[i + 1] = apk[i + 1]; mul2(kp[i], kp[i + 1], pe[i], pe[i + 1]);
                qp[i] = apq[i]; qp[i + 1] = apq[i + 1]; mul2(qp[i], qp[i + 1], pe[i], pe[i + 1]);
                kh[i] = ofr_k[i]; kh[i + 1] = ofr_k[i + 1]; mul2(kh[i], kh[i + 1], khe[i], khe[i + 1]);
            }
            if (NORM) {  // the state operands take the normalised rows
                mul2(kp[i], kp[i + 1], nk, nk);
                mul2(qp[i], qp[i + 1], nq, nq);
                mul2(kh[i], kh[i + 1], nk, nk);
            }
        }
        st_chunk(sm, SM_AP + sw_chunk(r, j, 128), apk);
        st_chunk(sm, SM_AP + sw_chunk(64 + r, j, 128), apq);
        st_chunk(sm, SM_APB + sw_chunk(r, j, 64), apb);
        if (MH) {  // off-tile A operand: rows 0..31 the K side, 32..63 the Q side
            st_chunk(sm, SM_OFF + sw_chunk(r - 32, j, 64), ofr_k);
            st_chunk(sm, SM_OFF + sw_chunk(r, j, 64), ofr_q);
        } else {   // off-tile B operand
            st_chunk(sm, SM_OFFB + sw_chunk(r, j, 32), ofr_k);
        }
        st_chunk(sm, SM_KQ + sw_chunk(r, j, 128), kp);
        st_chunk(sm, SM_KQ + sw_chunk(64 + r, j, 128), qp);
        st_chunk(sm, khb + tile_chunk(r, j), kh);  // the same layout: MMA4 reads it MN-major
    }
}

// Read the A/P tiles of TMEM lane quarter q (one warp) into A (fp32, strictly lower, rows scaled
// by beta) and the P operand (bf16, lower triangle). The diagonal tile (M = 128) holds row i of A
// (lanes 0..63) and of P (lanes 64..127); the off-diagonal tile (M = 64) holds its 64 rows in
// lanes 0..15 of each lane quarter: A rows 32..47, 48..63, then P rows 32..47, 48..63.
// NORM: the tiles were built from the raw rows; A_is takes nk_i nk_s and P_is takes nq_i nk_s
// (the inverse L2 norms of k and q rows, from the chunk's row sums of squares `nrm`).
template <bool NORM>
__device__ __forceinline__ void ap_readout(uint8_t *sm, float *As, uint32_t tmem_q, int q, int lane,
                                           const float *sbc, const float *nrm) {
    float vals[32];
    {
        const int L = 32 * q + lane;
        const int i = L & 63;
        const int j0 = (q & 1) ? 32 : 0;  // the diagonal half of row i
        tmem_ld32(tmem_q + TM_AP + j0, vals);
        tmem_ld_wait();
        if (NORM) {
            const float ri = row_inv_norm(nrm, L < 64 ? 0 : 1, i);
#pragma unroll
            for (int k = 0; k < 32; ++k) vals[k] *= ri * row_inv_norm(nrm, 0, j0 + k);
        }
        if (L < 64) {
            const float b = sbc[i];
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                float4 w;
                w.x = (j0 + k + 0 < i) ? vals[k + 0] * b : 0.f;
                w.y = (j0 + k + 1 < i) ? vals[k + 1] * b : 0.f;
                w.z = (j0 + k + 2 < i) ? vals[k + 2] * b : 0.f;
                w.w = (j0 + k + 3 < i) ? vals[k + 3] * b : 0.f;
                *reinterpret_cast<float4 *>(As + i * SA + j0 + k) = w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) vals[k] = (j0 + k <= i) ? vals[k] : 0.f;
            st_row32(sm + SM_P, i, j0, C, vals);
            if (j0 == 0) {
#pragma unroll
                for (int k = 0; k < 32; ++k) vals[k] = 0.f;
                st_row32(sm + SM_P, i, 32, C, vals);
            }
        }
    }
    tmem_ld32(tmem_q + TM_OFF, vals);
    tmem_ld_wait();
    if (lane < 16) {
        const int i = 32 + 16 * (q & 1) + lane;
        if (NORM) {
            const float ri = row_inv_norm(nrm, q < 2 ? 0 : 1, i);
#pragma unroll
            for (int k = 0; k < 32; ++k) vals[k] *= ri * row_inv_norm(nrm, 0, k);
        }
        if (q < 2) {
            const float b = sbc[i];
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4 *>(As + i * SA + k) =
                    make_float4(vals[k] * b, vals[k + 1] * b, vals[k + 2] * b, vals[k + 3] * b);
        } else {
            st_row32(sm + SM_P, i, 0, C, vals);
        }
    }
}

// (I + A)^{-1} on the 16 x 16 diagonal block w (one warp), by doubling: four 4 x 4 blocks in
// closed form, then 4 -> 8 -> 16 merges X21 = -X22 (A21 X11); then its block of T = X Diag(beta).
__device__ __forceinline__ void solve_diag_block(uint8_t *sm, const float *As, float *Xs, int warp, int lane,
                                                 const float *sbc) {
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
        for (int q = 0; q < 8; ++q) tv[q] = Xs[(B0 + r) * SA + B0 + h8 + q] * sbc[B0 + h8 + q];
        st_chunk(sm, SM_T + kmajor_offset(B0 + r, B0 + h8, C), tv);
    }
}

// Zero fills of the inverse (thread z of 128): the six strictly-upper 16 x 16 blocks of T. (The
// merges never read the upper blocks of X: they skip the K steps those blocks would contribute.)
__device__ __forceinline__ void solve_zero_fill(uint8_t *sm, int z) {
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

struct Maps {
    CUtensorMap q, k, g, v, o;
};

// Flags of a kernel instance:
// kGated: the g tensor holds logits x and the kernel forms g = -p.gate_bound * sigmoid(x).
// kNorm: q and k rows are divided by their L2 norms (sqrt(sum x^2 + 1e-6)) as they are read.
// kOutGate: O is multiplied by sigmoid(p.out_gate) before it is stored.
// kDump: (diagnostic) the CTA of the first (sequence, head) writes the chunkwise intermediates of
// its first p.dump_chunks chunks to p.dump (layout: kDumpFloatsPerChunk floats per chunk, see the
// stage offsets below); the plain path only.
// kOneRow: the operand build takes one row per loop iteration instead of two (the plain path only;
// same results bit for bit).
enum : int { kGated = 1, kNorm = 2, kOutGate = 4, kDump = 8, kOneRow = 16 };
constexpr int kDumpGam = 0, kDumpA = 64 * 128, kDumpT = kDumpA + 64 * 64, kDumpU = kDumpT + 64 * 64,
              kDumpS = kDumpU + 64 * 128, kDumpFloatsPerChunk = kDumpS + 128 * 128;

// The gate rows z (this head) of one chunk into the O staging tile, in the tile's own layout: a
// thread copies 8 of the 1024 16-byte chunks (row e / 16, channels 8 (e % 16) ..). Rows at or past
// `ln` (past the tensor end, never stored) get zeros.
__device__ __forceinline__ void stage_gate_rows(uint8_t *sm, const __nv_bfloat16 *zg, long long r0, int ln, int H,
                                                int h, int v, int dg) {
    uint4 z[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = v + 128 * i, row = e >> 4, cj = e & 15;
        z[i] = (row < ln && 8 * cj < dg)
                   ? __ldg(reinterpret_cast<const uint4 *>(zg + ((size_t)(r0 + row) * H + h) * dg + 8 * cj))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = v + 128 * i, row = e >> 4, cj = e & 15;
        *reinterpret_cast<uint4 *>(sm + SM_KQ + (cj >> 3) * 8192 + row * 128 + (((cj & 7) ^ (row & 7)) << 4)) = z[i];
    }
}

template <int F>
__global__ void __launch_bounds__(NTHREADS, 1)
    kda_prefill_tc_kernel(const __grid_constant__ Maps maps, const RunParams p) {
    constexpr bool GATED = (F & kGated) != 0, NORM = (F & kNorm) != 0, OGATE = (F & kOutGate) != 0;
    constexpr bool DUMP = (F & kDump) != 0;
    constexpr int ROWS = (F & kOneRow) ? 1 : 2;  // operand-build rows per loop iteration
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    float *wts = reinterpret_cast<float *>(sm + SM_WT);
    float *cst = reinterpret_cast<float *>(sm + SM_CST);
    float *gcs = reinterpret_cast<float *>(sm + SM_GC);
    float *sbeta = reinterpret_cast<float *>(sm + SM_BETA);
    float *nrmb = reinterpret_cast<float *>(sm + SM_NRM);
    float *As = reinterpret_cast<float *>(sm + SM_AS);
    float *Xs = reinterpret_cast<float *>(sm + SM_X);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM_BAR);
    uint32_t *tptr = reinterpret_cast<uint32_t *>(sm + SM_TPTR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H;
    const int dg = p.dk;  // head size in global memory (<= D; channels past it are zero here)
    const int h = blockIdx.x % H;
    const int n = p.order ? p.order[blockIdx.x / H] : (int)(blockIdx.x / H);

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
    int nchunks = (int)((eos - bos + C - 1) / C);
    if (p.max_chunks > 0 && nchunks > p.max_chunks) nchunks = p.max_chunks;
    if (p.skip && p.skip[(size_t)n * H + h]) return;

    if (warp == 0) {
        tmem_alloc(tptr, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int b = 0; b < BAR_N; ++b)
            mbar_init(&bars[b], b < BAR_OPS ? 1 : (b < BAR_SREADY ? NP : NS));
        fence_mbar_init();
    }
    if (NORM)  // the row-sum buffer of chunk 0 starts at zero (step 1 zeroes the later ones)
        for (int e = tid; e < 384; e += NTHREADS) nrmb[e] = 0.f;
    if (tid == 64) {
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.g);
        prefetch_tensormap(&maps.v);
        prefetch_tensormap(&maps.o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tptr;
    const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quarter

    if (warp == kIssuer) {
        // ---------------------------------------------------------------- issuer warp --------
        // The TMEM base as a warp-uniform value (lane 0's), so every MMA address is uniform.
        const uint32_t tmem = __shfl_sync(0xffffffffu, *tptr, 0);
        // The whole warp walks the chunks (one elected lane issues each MMA and copy) in the
        // order the work becomes ready: the chunk-parallel MMAs of chunk c (their operands come
        // from the prep warps), then the state chain of chunk c (MMA1, MMA2, MMA3/4) while the
        // prep warps already build chunk c + 1. Every K step is unrolled and its descriptor is a
        // constant step from the first. The g tiles after the first are fetched by the prep warps.
        auto wait = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(&bars[b], parity, kWaitNs));
        };
        bool iok = true;
        int last_g = -1, last_qk = -1, last_v = -1;  // chunk of the latest copy on each barrier
        auto load_g = [&](int cc) {
            const int r = (int)(bos + (long long)cc * C);
            if (elect_one()) {
                mbar_arrive_expect_tx(&bars[BAR_G], 16384);
                tma_load_3d(sm + SM_G, &maps.g, &bars[BAR_G], 0, h, r);
                tma_load_3d(sm + SM_G + 8192, &maps.g, &bars[BAR_G], 64, h, r);
            }
            __syncwarp();
            last_g = cc;
        };
        auto load_qk = [&](int cc) {
            const int r = (int)(bos + (long long)cc * C);
            if (elect_one()) {
                mbar_arrive_expect_tx(&bars[BAR_QK], 32768);
                for (int b = 0; b < 2; ++b) {
                    tma_load_3d(sm + SM_Q + 8192 * b, &maps.q, &bars[BAR_QK], 64 * b, h, r);
                    tma_load_3d(sm + SM_K + 8192 * b, &maps.k, &bars[BAR_QK], 64 * b, h, r);
                }
            }
            __syncwarp();
            last_qk = cc;
        };
        auto load_v = [&](int cc) {
            const int r = (int)(bos + (long long)cc * C);
            if (elect_one()) {
                mbar_arrive_expect_tx(&bars[BAR_V], 16384);
                tma_load_3d(sm + SM_VT, &maps.v, &bars[BAR_V], 0, h, r);
                tma_load_3d(sm + SM_VT + 8192, &maps.v, &bars[BAR_V], 64, h, r);
            }
            __syncwarp();
            last_v = cc;
        };
        // First-step descriptors of every operand.
        // K-major 128-byte-swizzled operands: K step st starts 32 B further in the 128-byte row,
        // and channels 64..127 (st >= 4) in the next atom column, R * 128 bytes on.
        auto ksw = [](int st, uint32_t rows) -> uint64_t {
            return (uint64_t)(((uint32_t)(st >> 2) * rows * 128u + (uint32_t)(st & 3) * 32u) >> 4);
        };
        const uint64_t d_ap = sdesc_sw128(sb + SM_AP, 16u, 1024u), d_apb = sdesc_sw128(sb + SM_APB, 16u, 1024u);
        const uint64_t d_offa = sdesc_sw128(sb + SM_OFF, 16u, 1024u), d_offb = sdesc_sw128(sb + SM_OFFB, 16u, 1024u);
        const uint64_t d_k = sdesc_sw128(sb + SM_KQ, 16u, 1024u), d_q = sdesc_sw128(sb + SM_KQ + 8192u, 16u, 1024u);
        const uint64_t d_v = sdesc_sw128(sb + SM_VT, 8192u, 1024u);
        const uint64_t d_t = sdesc(sb + SM_T, 128u, 1024u), d_p = sdesc(sb + SM_P, 128u, 1024u);
        const uint64_t d_kh0 = sdesc_sw128(sb + SM_KH, 8192u, 1024u);
        const uint64_t d_kh1 = sdesc_sw128(sb + SM_KH + 16384u, 8192u, 1024u);
        if (nchunks > 0) {
            load_g(0);
            load_qk(0);
            if (!p.zero_v) load_v(0);
        }
#pragma unroll 1
        for (int cc = 0; cc < nchunks; ++cc) {
            const uint32_t par = (uint32_t)(cc & 1);
            const bool more = cc + 1 < nchunks;
            // chunk-parallel part: the operands are built -> A/P tiles, and the q/k tiles are free
            // for the next chunk.
            if (!(iok = wait(BAR_OPS, par))) break;
            tc_fence_after();
#pragma unroll
            for (int st = 0; st < D / 16; ++st)
                mma_bf16_warp(tmem + TM_AP, d_ap + ksw(st, 128), d_apb + ksw(st, 64), idesc_bf16(128, 64), st > 0);
#pragma unroll
            for (int st = 0; st < D / 16; ++st)
                mma_bf16_warp(tmem + TM_OFF, d_offa + ksw(st, 64), d_offb + ksw(st, 32), idesc_bf16(64, 32), st > 0);
            mma_commit_warp(&bars[BAR_AP]);
            if (more) load_qk(cc + 1);
            // state chain. MMA1 = S^T [K+ ; Q+]^T from the bf16 state copy as soon as the operands
            // and the copy exist, the K+ half committed first ...
            if (!(iok = wait(BAR_SREADY, par))) break;
            tc_fence_after();
#pragma unroll
            for (int st = 0; st < D / 16; ++st)
                mma_bf16_tmem_a_warp(tmem + TM_D1, tmem + TM_SA + 8 * st, d_k + ksw(st, 128), idesc_bf16(128, 64),
                                     st > 0);
            mma_commit_warp(&bars[BAR_M1]);
#pragma unroll
            for (int st = 0; st < D / 16; ++st)
                mma_bf16_tmem_a_warp(tmem + o_slot(cc), tmem + TM_SA + 8 * st, d_q + ksw(st, 128), idesc_bf16(128, 64),
                                     st > 0);
            mma_commit_warp(&bars[BAR_M1Q]);
            // ... U^T = V^T T^T - (K+ S)^T T^T once T exists and -(K+ S)^T has been read out of
            // TM_D1, which U^T then takes over (V tile as an MN-major A operand, skipped for v = 0;
            // the second product reads -(K+ S)^T from TMEM) ...
            if (!(iok = wait(BAR_TREADY, par))) break;
            if (!(iok = wait(BAR_RREADY, par))) break;
            if (!p.zero_v && !(iok = wait(BAR_V, par))) break;
            tc_fence_after();
            if (!p.zero_v) {
#pragma unroll
                for (int st = 0; st < C / 16; ++st)
                    mma_bf16_warp(tmem + TM_D1, d_v + kDescStepMN128 * st, d_t + kDescStepKmajor * st,
                                  idesc_bf16(128, 64) | kIdescAMajorMN, st > 0);
            }
#pragma unroll
            for (int st = 0; st < C / 16; ++st)
                mma_bf16_tmem_a_warp(tmem + TM_D1, tmem + TM_RA + 8 * st, d_t + kDescStepKmajor * st,
                                     idesc_bf16(128, 64), (!p.zero_v || st > 0) ? 1u : 0u);
            mma_commit_warp(&bars[BAR_M2]);
            if (more && !p.zero_v) {  // the v tile is consumed: fetch the next one
                if (!(iok = wait(BAR_M2, par))) break;
                load_v(cc + 1);
            }
            // ... then O^T += U^T P^T and S^T += U^T Khat.
            if (!(iok = wait(BAR_UREADY, par))) break;
            tc_fence_after();
#pragma unroll
            for (int st = 0; st < C / 16; ++st)
                mma_bf16_tmem_a_warp(tmem + o_slot(cc), tmem + TM_RA + 8 * st, d_p + kDescStepKmajor * st,
                                     idesc_bf16(128, 64), 1u);
            const uint64_t d_kh = par ? d_kh1 : d_kh0;
#pragma unroll
            for (int st = 0; st < C / 16; ++st)
                mma_bf16_tmem_a_warp(tmem + TM_S, tmem + TM_RA + 8 * st, d_kh + kDescStepMN128 * st,
                                     idesc_bf16(128, 128) | kIdescBMajorMN, 1u);
            mma_commit_warp(&bars[BAR_M34]);
        }
        if (!iok) {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            // Drain what was issued (bounded), so no MMA or copy is in flight at exit. At most one
            // copy per TMA barrier is outstanding, so its phase parity is its chunk's.
            mma_commit_warp(&bars[BAR_DRAIN]);
            (void)mbar_wait(&bars[BAR_DRAIN], 0, kWaitNs);
            if (last_g >= 0) (void)mbar_wait(&bars[BAR_G], (uint32_t)(last_g & 1), kWaitNs);
            if (last_qk >= 0) (void)mbar_wait(&bars[BAR_QK], (uint32_t)(last_qk & 1), kWaitNs);
            if (last_v >= 0) (void)mbar_wait(&bars[BAR_V], (uint32_t)(last_v & 1), kWaitNs);
        }
        __syncwarp();
    } else if (warp >= kStateWarp0) {
        // --------------------------------------------------------------- state warps --------
        // Thread v = TMEM lane v = value column v of the state. Per chunk: bf16 copy of S for
        // MMA1, S <- S Diag(gam_last), -(K+ S)^T and U^T as bf16 A operands, O write-back.
        const int v = tid - NP;
        __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o);
        bool ok = true;
        const long long init_off = p.init ? state_slot_offset(p.init_idx, p.pool, n, H, h, dg, p.err) : -1;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {  // initial state -> TMEM (fp32)
            const int k0 = 32 * cb;
            float buf[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                buf[i] = p.identity_init ? (k0 + i == v ? 1.f : 0.f)
                                         : ((init_off >= 0 && v < dg && k0 + i < dg)
                                                ? __ldcs(p.init + init_off + (size_t)(k0 + i) * dg + v)
                                                : 0.f);
            tmem_st32(tmem + tq + TM_S + k0, buf);
        }
        tmem_st_wait();

        // O of a finished chunk (TMEM columns TM_D1 + 64 ..+63 = its 64 tokens) straight to
        // global memory: each warp store covers 32 consecutive value columns (64 bytes).
        const __nv_bfloat16 *zg = static_cast<const __nv_bfloat16 *>(p.out_gate);
        auto store_o = [&](const float (&o0)[32], const float (&o1)[32], long long r0, int ln) {
            if (v >= dg) return;  // a padded value column: nothing to store
            __nv_bfloat16 *dst = og + ((size_t)r0 * H + h) * dg + v;
            const size_t rs = (size_t)H * dg;  // elements between consecutive tokens
            if (OGATE) {  // a ragged chunk: gate each stored element
                const __nv_bfloat16 *zr = zg + ((size_t)r0 * H + h) * dg + v;
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs, zr += rs)
                    if (r < ln) *dst = __float2bfloat16_rn(o0[r] * __fdividef(1.f, 1.f + ex2(-__bfloat162float(*zr) * kLog2e)));
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs, zr += rs)
                    if (32 + r < ln) *dst = __float2bfloat16_rn(o1[r] * __fdividef(1.f, 1.f + ex2(-__bfloat162float(*zr) * kLog2e)));
            } else if (ln == C) {
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs) *dst = __float2bfloat16_rn(o0[r]);
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs) *dst = __float2bfloat16_rn(o1[r]);
            } else {
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs)
                    if (r < ln) *dst = __float2bfloat16_rn(o0[r]);
#pragma unroll
                for (int r = 0; r < 32; ++r, dst += rs)
                    if (32 + r < ln) *dst = __float2bfloat16_rn(o1[r]);
            }
        };

        // O of chunk cc (its TMEM slot) out. A chunk that is full (or ends the tensor: rows past its
        // end are not written) goes through the [K+ ; Q+] region (free from MMA1 of the next chunk
        // until the prep warps build the chunk after it) in the TMA tile layout, one bulk tensor
        // store per 64 channels, after which the region is released to the prep warps (KQFREE). A
        // ragged chunk that does not end the tensor takes plain stores, so rows of the next
        // sequence are never written.
        const long long total_rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
        auto flush_o = [&](int cc, long long r0, int ln) {
            if (ln == C || r0 + ln >= total_rows) {
                // The warp's 32 value columns x 64 tokens in the MMA-fragment layout, bf16 pairs of
                // consecutive tokens, stored transposed by stmatrix straight into the TMA tile
                // layout (16 bytes = 8 value columns of one token per row of each matrix).
                const uint32_t lq = (uint32_t)(32 * (warp & 3));
                uint32_t f0[32], f1[32];
                tmem_ld_frag64(tmem + (lq << 16) + o_slot(cc), f0);
                tmem_ld_frag64(tmem + ((lq + 16) << 16) + o_slot(cc), f1);
                tmem_ld_wait();
                const int i4 = lane >> 3, jr = lane & 7;
                const int cj = (int)((lq + 16 * (i4 >> 1) + 8 * (i4 & 1)) >> 3);  // 8-column chunk of matrix i4
                const uint32_t abase = sb + SM_KQ + (uint32_t)((cj >> 3) * 8192);
                if (OGATE) {
                    // z into the tile first; each O value is scaled by sigmoid(z) read back in the
                    // same fragment layout, so O is rounded to bf16 once.
                    stage_gate_rows(sm, zg, r0, (int)min((long long)C, total_rows - r0), H, h, v, dg);
                    state_sync();
                }
                auto gate = [&](float x, float z) { return x * __fdividef(1.f, 1.f + ex2(-z * kLog2e)); };
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int tok = 8 * k + jr;
                    const uint32_t addr = abase + (uint32_t)(tok * 128 + (((cj & 7) ^ (tok & 7)) << 4));
                    float a0 = __uint_as_float(f0[4 * k]), a1 = __uint_as_float(f0[4 * k + 1]);
                    float b0 = __uint_as_float(f0[4 * k + 2]), b1 = __uint_as_float(f0[4 * k + 3]);
                    float c0 = __uint_as_float(f1[4 * k]), c1 = __uint_as_float(f1[4 * k + 1]);
                    float d0 = __uint_as_float(f1[4 * k + 2]), d1 = __uint_as_float(f1[4 * k + 3]);
                    if (OGATE) {
                        uint32_t za, zb, zc, zd;
                        ldmatrix_x4_trans(addr, za, zb, zc, zd);
                        a0 = gate(a0, bf_lo(za)); a1 = gate(a1, bf_hi(za));
                        b0 = gate(b0, bf_lo(zb)); b1 = gate(b1, bf_hi(zb));
                        c0 = gate(c0, bf_lo(zc)); c1 = gate(c1, bf_hi(zc));
                        d0 = gate(d0, bf_lo(zd)); d1 = gate(d1, bf_hi(zd));
                    }
                    stmatrix_x4_trans(addr, pack_bf16(a0, a1), pack_bf16(b0, b1), pack_bf16(c0, c1), pack_bf16(d0, d1));
                }
                fence_async_smem();
                state_sync();
                if (v == 0) {
                    tma_store_3d(&maps.o, sm + SM_KQ, 0, h, (int)r0);
                    tma_store_3d(&maps.o, sm + SM_KQ + 8192, 64, h, (int)r0);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                return;
            }
            float o0[32], o1[32];
            tmem_ld32(tmem + tq + o_slot(cc), o0);
            tmem_ld32(tmem + tq + o_slot(cc) + 32, o1);
            tmem_ld_wait();
            store_o(o0, o1, r0, ln);
        };
        long long prev_row0 = 0;
        int prev_len = 0;
        int c = 0;
#pragma unroll 1
        for (; c < nchunks; ++c) {
            const uint32_t par = (uint32_t)(c & 1);
            const long long row0 = bos + (long long)c * C;
            const int len = (int)min((long long)C, eos - row0);
            if (OGATE && (v >> 1) < len && 64 * (v & 1) < dg)  // this chunk's gate rows into L2 (read when its O is written)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(zg + ((size_t)(row0 + (v >> 1)) * H + h) * dg + 64 * (v & 1)));
            // The state after chunk c - 1 (MMA4) and gam_last of chunk c (its step 1).
            if (c > 0 && !(ok = state_wait(&bars[BAR_M34], par ^ 1u))) break;
            if (!(ok = state_wait(&bars[c & 1 ? BAR_S1D1 : BAR_S1D0], (uint32_t)((c >> 1) & 1)))) break;
            tc_fence_after();
            // One pass over the state: its bf16 copy for MMA1, and S <- S Diag(gam_last) for MMA4.
            {
                const float *gc = gcs + 128 * (c % 3);
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    float sv[32];
                    tmem_ld32(tmem + tq + TM_S + 32 * cb, sv);
                    tmem_ld_wait();
                    if (DUMP && blockIdx.x == 0 && c < p.dump_chunks) {  // S at the chunk start, [d_k][d_v]
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            p.dump[(size_t)c * kDumpFloatsPerChunk + kDumpS + (32 * cb + i) * D + v] = sv[i];
                    }
                    uint32_t w[16];
                    pack32(sv, w, 1.f);
                    tmem_st16(tmem + tq + TM_SA + 16 * cb, w);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float gv[8];
                        lds8(gv, gc + 32 * cb + i);
#pragma unroll
                        for (int t = 0; t < 8; t += 2) mul2(sv[i + t], sv[i + t + 1], gv[t], gv[t + 1]);
                    }
                    tmem_st32(tmem + tq + TM_S + 32 * cb, sv);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(&bars[BAR_SREADY]);

            // A and P out of TMEM and the 16 x 16 diagonal blocks of (I + A)^{-1}; the prep warps
            // merge the blocks once EPIDONE is signalled. P and T are rewritten only after MMA2 and
            // MMA3 of the previous chunk (M34 above).
            if (!(ok = state_wait(&bars[BAR_AP], par))) break;
            tc_fence_after();
            {
                const float *sbc = sbeta + 64 * par;
                ap_readout<NORM>(sm, As, tmem + tq, warp & 3, lane, sbc, nrmb + 128 * (c % 3));
                state_sync();
                if (DUMP && blockIdx.x == 0 && c < p.dump_chunks)  // A (strictly lower, beta-scaled rows)
                    for (int e = v; e < 64 * 64; e += NS) {
                        const int r = e >> 6, s2 = e & 63;
                        p.dump[(size_t)c * kDumpFloatsPerChunk + kDumpA + e] = s2 < r ? As[r * SA + s2] : 0.f;
                    }
                solve_diag_block(sm, As, Xs, warp & 3, lane, sbc);
                solve_zero_fill(sm, v);
            }
            fence_async_smem();  // T and P are read by MMAs
            mbar_arrive(&bars[BAR_EPIDONE]);

            if (!(ok = state_wait(&bars[BAR_M1], par))) break;
            tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float ks[32];
                tmem_ld32(tmem + tq + TM_D1 + 32 * hh, ks);
                tmem_ld_wait();
                uint32_t w[16];
                pack32(ks, w, -1.f);
                tmem_st16(tmem + tq + TM_RA + 16 * hh, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[BAR_RREADY]);

            // O of the previous chunk, while the prep warps merge the inverse: staged in the
            // [K+ ; Q+] region once MMA1 of this chunk has read it.
            if (!(ok = state_wait(&bars[BAR_M1Q], par))) break;
            tc_fence_after();
            if (c > 0) flush_o(c - 1, prev_row0, prev_len);
            mbar_arrive(&bars[BAR_KQFREE]);

            if (!(ok = state_wait(&bars[BAR_M2], par))) break;
            tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float u[32];
                tmem_ld32(tmem + tq + TM_D1 + 32 * hh, u);
                tmem_ld_wait();
                if (DUMP && blockIdx.x == 0 && c < p.dump_chunks) {  // U, [token][d_v]
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        p.dump[(size_t)c * kDumpFloatsPerChunk + kDumpU + (32 * hh + i) * D + v] = u[i];
                }
                uint32_t w[16];
                pack32(u, w, 1.f);
                tmem_st16(tmem + tq + TM_RA + 16 * hh, w);  // U^T replaces -(K+ S)^T (MMA2 has finished)
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[BAR_UREADY]);
            prev_row0 = row0;
            prev_len = len;
        }
        if (ok && nchunks > 0) {  // O of the last chunk
            ok = state_wait(&bars[BAR_M34], (uint32_t)((nchunks - 1) & 1));
            if (ok) {
                tc_fence_after();
                flush_o(nchunks - 1, prev_row0, prev_len);
            }
        }
        if (v == 0) bulk_wait_all();  // every O store is complete (and has read shared memory)
        if (ok) {
            const long long fin_off = p.fin ? state_slot_offset(p.fin_idx, p.pool, n, H, h, dg, p.err) : -1;
            if (fin_off >= 0 && v < dg) {
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    float sv[32];
                    tmem_ld32(tmem + tq + TM_S + 32 * cb, sv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (32 * cb + i < dg) __stcs(p.fin + fin_off + (size_t)(32 * cb + i) * dg + v, sv[i]);
                }
            }
        } else if (v == 0) {
            atomicOr(p.err, kErrTimeout);
        }
    } else {
        // ---------------------------------------------------------------- prep warps --------
        // Everything of a chunk that does not depend on the state: Gam, the decay-scaled
        // operands, the A/P tiles, T = (I + A)^{-1} Diag(beta). Chunk c + 1 is built here while
        // the state warps and the issuer run the state chain of chunk c.
        const __nv_bfloat16 *bg = static_cast<const __nv_bfloat16 *>(p.beta);
        bool ok = true;
        // Thread mapping: channels 8j..8j+7 (j = 8 * (warp >> 2) + lane % 8, the fastest index
        // across lanes), rows tr0 .. tr0 + 3 with tr0 = 16 * (warp % 4) + 4 * (lane / 8).
        const int j = 8 * (warp >> 2) + (lane & 7);
        const int rq = lane >> 3;
        const int rb = warp & 3;  // 16-row block
        const int tr0 = 16 * rb + 4 * rq;
        const int mh = rb >> 1;
        float gm[4][8];  // Gam_r - Gam_ref of the thread's 4 rows x 8 channels (current chunk; ref = row 15 or 47)
        int g_inflight = -1;  // chunk of a g-tile copy issued here and not yet waited for
        // beta of token tid of a chunk, loaded one step ahead (raw bf16 bits, converted when used)
        auto load_beta = [&](int cc) -> uint32_t {
            const long long r0 = bos + (long long)cc * C;
            if (tid < C && r0 + tid < eos)
                return *reinterpret_cast<const uint16_t *>(bg + (size_t)(r0 + tid) * H + h);
            return 0u;
        };
        uint32_t beta_next = nchunks > 0 ? load_beta(0) : 0u;
        // Step 1 of chunk cc: wait for its g tile, Gam = cumsum of g into gm, the reference rows
        // and per-channel factors into shared memory, beta into its sbeta buffer; then fetch the
        // next g tile. Runs while the A/P MMAs of chunk cc - 1 are in flight. False if a wait ran
        // out.
        auto step1 = [&](int cc) -> bool {
            const long long r0 = bos + (long long)cc * C;
            const int ln = (int)min((long long)C, eos - r0);
            QKRows qk;
            if (NORM) {  // in flight while the cumsum runs
                load_qk_rows(qk, static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
                             r0, ln, H, h, tr0, j, p.dk);
                if (tid < 128) nrmb[128 * ((cc + 1) % 3) + tid] = 0.f;
            }
            const float bet = __uint_as_float(beta_next << 16);
            if (cc + 1 < nchunks) beta_next = load_beta(cc + 1);
            if (!prep_wait(&bars[BAR_G], (uint32_t)(cc & 1))) return false;
            g_inflight = -1;

            // ---- 1. Gam = cumsum_r g within the chunk, per key channel --------------------------
            // A thread's own 4 rows in registers, then across the 4 lanes of a 16-row block (two
            // shuffle steps), then across the four blocks through shared memory.
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = tr0 + m;
                const uint4 w = *reinterpret_cast<const uint4 *>(sm + SM_G + tile_chunk(r, j));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float x = (i & 1) ? bf_hi(ww[i >> 1]) : bf_lo(ww[i >> 1]);
                    if (GATED) x = __fdividef(-p.gate_bound, 1.f + ex2(-x * kLog2e));  // scaled sigmoid
                    x = r < ln ? x : 0.f;
                    gm[m][i] = m ? gm[m - 1][i] + x : x;
                }
            }
            {
                float incl[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) incl[i] = gm[3][i];
#pragma unroll
                for (int d = 8; d < 32; d <<= 1) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float t = __shfl_up_sync(0xffffffffu, incl[i], d);
                        if (lane >= d) incl[i] += t;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float excl = incl[i] - gm[3][i];
#pragma unroll
                    for (int m = 0; m < 4; ++m) gm[m][i] += excl;
                }
                if (rq == 3) {  // the 16-row block's sums
                    *reinterpret_cast<float4 *>(wts + 128 * rb + 8 * j) = make_float4(incl[0], incl[1], incl[2], incl[3]);
                    *reinterpret_cast<float4 *>(wts + 128 * rb + 8 * j + 4) = make_float4(incl[4], incl[5], incl[6], incl[7]);
                }
                // gm now holds Gam relative to the start of the thread's 16-row block. The operand
                // build needs Gam_r - Gam_ref with the reference row at the end of block 0 or 2
                // (rows 15, 47): for blocks 1 and 3 that is the block-relative value itself, for
                // blocks 0 and 2 the block-relative value minus the block's total (held by the
                // lanes of row group 3).
                if ((rb & 1) == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float tot = __shfl_sync(0xffffffffu, incl[i], (lane & 7) | 24);
#pragma unroll
                        for (int m = 0; m < 4; ++m) gm[m][i] -= tot;
                    }
                }
            }
            if (tid < C) sbeta[64 * (cc & 1) + tid] = bet;
            if (NORM) add_row_square_sums(nrmb + 128 * (cc % 3), qk, tr0, lane);
            prep_sync();
            if (tid == 0 && cc + 1 < nchunks) {  // every prep thread has read the g tile
                const int r = (int)(bos + (long long)(cc + 1) * C);
                mbar_arrive_expect_tx(&bars[BAR_G], 16384);
                tma_load_3d(sm + SM_G, &maps.g, &bars[BAR_G], 0, h, r);
                tma_load_3d(sm + SM_G + 8192, &maps.g, &bars[BAR_G], 64, h, r);
                g_inflight = cc + 1;
            }
            if (DUMP && blockIdx.x == 0 && cc < p.dump_chunks) {  // Gam, [token][d_k]
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        p.dump[(size_t)cc * kDumpFloatsPerChunk + kDumpGam + (tr0 + m) * D + 8 * j + i] =
                            gm[m][i] + (mh ? wts[8 * j + i] + wts[128 + 8 * j + i] + wts[256 + 8 * j + i] : wts[8 * j + i]);
            }
            if (NORM && tid < 128) {  // the row sums of squares are complete: inverse norms in place
                float *nb = nrmb + 128 * (cc % 3) + tid;
                *nb = rsqrtf(*nb + 1e-6f);
            }
            if (tid < 128) {
                const int ch = tid;
                const float G15 = wts[ch], G31 = G15 + wts[128 + ch];
                const float G47 = G31 + wts[256 + ch], G63 = G47 + wts[384 + ch];
                cst[CST_C0 * 128 + ch] = ex2((G31 - G15) * kLog2e);
                cst[CST_C1 * 128 + ch] = ex2((G47 - G31) * kLog2e);
                cst[CST_EM0 * 128 + ch] = ex2(G15 * kLog2e);
                cst[CST_EG31 * 128 + ch] = ex2(G31 * kLog2e);
                cst[CST_E63M1 * 128 + ch] = ex2((G63 - G47) * kLog2e);
                cst[CST_E63G31 * 128 + ch] = ex2((G63 - G31) * kLog2e);
                gcs[128 * (cc % 3) + ch] = ex2(G63 * kLog2e);
            }
            // No group barrier here: every prep thread arrives after its own writes, so the phase
            // completes only when all of them are visible; the operand build of chunk cc reads
            // the factors after the group barriers of the waits and merges in between.
            mbar_arrive(&bars[(cc & 1) ? BAR_S1D1 : BAR_S1D0]);  // gam_last and beta of chunk cc are in place
            return true;
        };

        if (nchunks > 0) ok = step1(0);
#pragma unroll 1
        for (int c = 0; ok && c < nchunks; ++c) {
            const uint32_t par = (uint32_t)(c & 1);
            const long long row0 = bos + (long long)c * C;
            const int len = (int)min((long long)C, eos - row0);

            // ---- 2. decay-scaled operands (once MMA1 of the previous chunk has read [K+ ; Q+]) --
            if (!(ok = prep_wait(&bars[BAR_QK], par, c > 0 ? &bars[BAR_KQFREE] : nullptr, par ^ 1u))) break;
            if (mh)
                build_operands<1, NORM, ROWS>(sm, gm, cst, tr0, j, len, SM_KH + 16384u * par, nrmb + 128 * (c % 3));
            else
                build_operands<0, NORM, ROWS>(sm, gm, cst, tr0, j, len, SM_KH + 16384u * par, nrmb + 128 * (c % 3));
            fence_async_smem();
            mbar_arrive(&bars[BAR_OPS]);

            // ---- step 1 of the next chunk while the A/P MMAs run --------------------------------
            if (c + 1 < nchunks && !(ok = step1(c + 1))) break;
            const float *sbc = sbeta + 64 * par;  // beta of this chunk

            // ---- 3. X = (I + A)^{-1}, written to T = X Diag(beta) as it completes ---------------
            // The state warps have read A and P out of TMEM and inverted the 16 x 16 diagonal
            // blocks (with the zero fills); the block merges run here.
            if (!(ok = prep_wait(&bars[BAR_EPIDONE], par))) break;
            // (b) 16 -> 32: warp (p, nt) < 4 computes column tile nt of X_{2p+1,2p} (tf32 mma).
            // Meanwhile warps 4..7 start (c)'s first product Y = A_BA X_AA with what the 16 x 16
            // blocks already give: its columns 16..31 whole (X_AA is zero above X_11 there) and the
            // first half (X_00) of its columns 0..15, finished with X_10 once (b) is done.
            float *Yc = reinterpret_cast<float *>(sm + SM_YC);
            float accp[4];
            const int w4 = warp - 4, cmt = w4 >> 1, cnt = w4 & 1;  // (c) tiles of warps 4..7
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
                store_t_16x8(sm + SM_T, 16 * I, 16 * J + 8 * nt, acc, sbc, lane);
            } else {
                float acc[4];
                const float *Ab = As + (32 + 16 * cmt) * SA;
                warp_mma_16x8<16>(acc, Ab + 16, SA, Xs + 16 * SA + 8 * (2 + cnt), SA, lane);
                warp_store_16x8(Yc + 16 * cmt * SA + 8 * (2 + cnt), SA, acc, 1.f, lane);
                warp_mma_16x8<16>(accp, Ab, SA, Xs + 8 * cnt, SA, lane);
            }
            prep_sync();
            if (warp >= 4) {  // the rest of (c)'s columns 0..15: + A_BA[:, 16..31] X_10
                warp_mma_16x8<16, false>(accp, As + (32 + 16 * cmt) * SA + 16, SA, Xs + 16 * SA + 8 * cnt, SA, lane);
                warp_store_16x8(Yc + 16 * cmt * SA + 8 * cnt, SA, accp, 1.f, lane);
            }
            prep_sync();
            // (c) 32 -> 64: X_BA = -X_BB Y with 32 x 32 blocks; warp w owns one 16 x 8 tile. X_BB is
            // zero above X_33, so its first 16 rows take K = 16.
            {
                const int mt = warp >> 2, nt = warp & 3;
                float acc[4];
                if (mt == 0)
                    warp_mma_16x8<16>(acc, Xs + 32 * SA + 32, SA, Yc + 8 * nt, SA, lane);
                else
                    warp_mma_16x8<32>(acc, Xs + 48 * SA + 32, SA, Yc + 8 * nt, SA, lane);
                store_t_16x8(sm + SM_T, 32 + 16 * mt, 8 * nt, acc, sbc, lane);
            }
            fence_async_smem();  // the T stores
            mbar_arrive(&bars[BAR_TREADY]);
            if (DUMP && blockIdx.x == 0 && c < p.dump_chunks) {  // T = (I + A)^{-1} Diag(beta), [token][token]
                prep_sync();
                for (int e = tid; e < 64 * 64; e += NP) {
                    const int r = e >> 6, s2 = e & 63;
                    p.dump[(size_t)c * kDumpFloatsPerChunk + kDumpT + e] =
                        __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + SM_T + kmajor_offset(r, s2, C)));
                }
            }
        }
        if (!ok && tid == 0) {
            atomicOr(p.err, kErrTimeout);
            if (g_inflight >= 0) (void)mbar_wait(&bars[BAR_G], (uint32_t)(g_inflight & 1), kWaitNs);
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

bool encode_map(CUtensorMap *map, const void *base, long long rows, int H, int d) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_row_tile_map(CUtensorMap *map, const void *base, long long rows, int H, int d) {
    return encode_map(map, base, rows, H, d);
}

// bf16 with d_k == d_v in {32, 64, 128}: smaller heads run the d = 128 kernel with the missing
// channels zero (the tensor maps read them as zeros, the stores skip them), when the driver encodes
// their tensor maps.
bool tc_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p) {
    if (dtype != KDA_BF16 || dk != dv || (dk != 32 && dk != 64 && dk != D)) return false;
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    if (rows <= 0 || rows > 0x7fffffffLL - C) return false;
    if (!tensor_map_encoder()) return false;
    CUtensorMap probe;
    return encode_map(&probe, p.q, rows, p.H, dk);
}

// One instance per combination of the flags, indexed by them; then the diagnostic instance and the
// plain instance with the one-row operand build.
constexpr int kNumTcKernels = 10;
const void *const kTcKernels[kNumTcKernels] = {
    (const void *)kda_prefill_tc_kernel<0>, (const void *)kda_prefill_tc_kernel<1>,
    (const void *)kda_prefill_tc_kernel<2>, (const void *)kda_prefill_tc_kernel<3>,
    (const void *)kda_prefill_tc_kernel<4>, (const void *)kda_prefill_tc_kernel<5>,
    (const void *)kda_prefill_tc_kernel<6>, (const void *)kda_prefill_tc_kernel<7>,
    (const void *)kda_prefill_tc_kernel<kDump>, (const void *)kda_prefill_tc_kernel<kOneRow>};

cudaError_t launch_tc_prefill(const RunParams &p, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[256] = {};
    static int sm_count[256] = {};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            for (int f = 0; f < kNumTcKernels && e == cudaSuccess; ++f)
                e = cudaFuncSetAttribute(kTcKernels[f], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
        sms = sm_count[dev];
    }
    const long long rows = p.cu_seqlens ? (long long)p.T : (long long)p.n_seqs * p.T;
    Maps maps;
    if (!encode_map(&maps.q, p.q, rows, p.H, p.dk) || !encode_map(&maps.k, p.k, rows, p.H, p.dk) ||
        !encode_map(&maps.g, p.g, rows, p.H, p.dk) || !encode_map(&maps.v, p.v, rows, p.H, p.dk) ||
        !encode_map(&maps.o, p.o, rows, p.H, p.dk))
        return cudaErrorInvalidValue;
    int f = p.dump ? 8 : (p.gate_bound > 0.f ? kGated : 0) | (p.qk_l2norm ? kNorm : 0) | (p.out_gate ? kOutGate : 0);
    const long long grid = (long long)p.n_seqs * p.H;
    // With more CTAs than SMs every SM runs one and the smaller build code is faster (64 packed
    // sequences: 6.75 against 7.16 ms); with fewer, the two-row build (B=4 T=8192 H=32: 0.546
    // against 0.553 ms).
    if (f == 0 && grid > sms) f = 9;
    void *args[] = {(void *)&maps, (void *)&p};
    return cudaLaunchKernel(kTcKernels[f], dim3((unsigned)grid), dim3(NTHREADS), args, SMEM_BYTES, s);
}

}  // namespace kda
