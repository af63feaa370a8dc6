// kda_prefill_tf32.cu -- chunked KDA prefill for fp32 inputs with heads of up to 64 channels, on
// the sm_103a tensor cores in tf32 (tcgen05 kind::tf32, fp32 accumulation in TMEM).
//
// What is computed: the same chunkwise form of the KDA recurrence as kda_prefill_tc.cu ("Inside
// Kimi K3's Architecture" (maidul-haque blog), "Kimi Delta Attention: the linear core"; "Kimi K3
// Explained" (researchpapers.dev), "Architecture at a glance": with the log-decay bounded below,
// every causal tile of the chunkwise computation is a dense tensor-core matmul). Per chunk of
// C = 64 tokens, with S the d_k x d_v state at the chunk start and Gam the per-channel cumsum of g:
//     A = strict_lower(Diag(beta) (K*gam)(K/gam)^T),  P = lower((Q*gam)(K/gam)^T)
//     T = (I + A)^{-1} Diag(beta),  U = T (V - (K*gam) S),  O = (Q*gam) S + P U
//     S <- Diag(gam_last) S + (K*gam_last/gam)^T U
// A and P come from three 32 x 32 tiles whose decay factors stay inside fp32 (reference rows
// Gam_15, Gam_47 for the diagonal halves, Gam_31 for the off-diagonal tile), exactly as in the
// bf16 kernel; K+ = K exp(Gam_r), Q+ = Q exp(Gam_r) and Khat = K exp(Gam_last - Gam_r) are single
// products with a factor of at most 1.
//
// Precision: every product runs on the tensor cores with tf32 operands (10-bit mantissa, rounded
// to nearest when the operands are written) and fp32 accumulation; the state stays fp32 in TMEM
// and is itself the A operand of MMA1 (a tf32 MMA reads fp32 words). The triangular inverse is a
// plain fp32 forward substitution. Everything else is fp32 on the CUDA cores.
//
// Layout of the work: one CTA of 256 threads per (sequence, head), chunks in order, the steps of a
// chunk one after another between block barriers (the path is meant for the small fp32
// configurations, where a chunk's latency, not throughput, is what counts); the only overlap
// between chunks is step 1 of the next chunk (Gam, its factors, beta), which runs while MMA1 of the
// current one is in flight.
// Heads of 32 channels run with the missing channels zero (zero key and query channels add
// nothing; the padded state rows and columns stay zero and are not stored). The state lives in
// TMEM lanes 0..63 (value columns); lanes 64..127 hold zeros so that the M = 128 MMAs stay in
// their simplest layout. All shared-memory operands are K-major without swizzle (8-row x 16-byte
// core matrices), which a tf32 MMA reads for both operands.
// Every mbarrier wait is bounded; on time-out the CTA records kErrTimeout and leaves the loop.
#include <mutex>

#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;        // chunk length
constexpr int DP = 64;       // padded head size (d_k == d_v <= 64)
constexpr int NT = 256;      // threads
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitNs = 1000000000ull;

// Shared memory (bytes from a 1024-byte aligned base). Operand tiles: fp32 words, K-major, no
// swizzle, 64 K-elements per row (256 B): element (r, k) at tk_off(r, k).
constexpr uint32_t SM_APA = 0;                    // [K*f ; Q*f]          128 rows
constexpr uint32_t SM_APB = SM_APA + 32768;       // K/f                   64 rows
constexpr uint32_t SM_OFFA = SM_APB + 16384;      // off tile A: K*e (rows 32..63) ; Q*e (rows 32..63)
constexpr uint32_t SM_OFFB = SM_OFFA + 16384;     // off tile B: K*e' (rows 0..31)   32 rows
constexpr uint32_t SM_KQ = SM_OFFB + 8192;        // [K+ ; Q+]            128 rows
constexpr uint32_t SM_KHT = SM_KQ + 32768;        // Khat^T: row = key channel, K = token
constexpr uint32_t SM_VT = SM_KHT + 16384;        // V^T: row = value column (rows 64..127 zero), K = token
constexpr uint32_t SM_T = SM_VT + 32768;          // T: row r, K = s
constexpr uint32_t SM_P = SM_T + 16384;           // P: row r, K = s
constexpr uint32_t SG = 68;                       // row stride (floats) of Gam: bank-free for the build's lanes
constexpr uint32_t SM_GAM = SM_P + 16384;         // Gam, fp32 [64 rows][SG]
constexpr uint32_t SA = 68;                       // row stride (floats) of A and X
constexpr uint32_t SM_AS = SM_APA;                //   A (fp32 [64][SA], beta-scaled rows) once the A/P MMAs are done
constexpr uint32_t SM_X = SM_APA + 64 * SA * 4;   //   X = (I + A)^{-1}, the same time
constexpr uint32_t SM_CST = SM_GAM + 64 * SG * 4;  // per-channel factors [chunk parity][CST_N][64]
constexpr uint32_t SM_WS = SM_CST + 4096;         // block sums of g [4][64]
constexpr uint32_t SM_BETA = SM_WS + 1024;        // beta [64]
constexpr uint32_t SM_BAR = SM_BETA + 256;        // mbarrier
constexpr uint32_t SM_TPTR = SM_BAR + 16;         // TMEM base address
constexpr uint32_t SM_USED = SM_TPTR + 16;
constexpr uint32_t SMEM_BYTES = SM_USED + 1024;   // + alignment slack
static_assert(SM_X + 64 * SA * 4 <= SM_OFFA, "solve buffers overflow the A/P operand tiles");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

enum { CST_M0 = 0, CST_M1, CST_C0, CST_C1, CST_GL, CST_GAML, CST_N };  // CST_GL: Gam_last*log2e, CST_GAML: exp(Gam_last)
static_assert(CST_N * 256 <= 2048, "factor rows overflow");

// TMEM columns.
constexpr uint32_t TM_AP = 0, TM_OFF = 64, TM_RA = 128, TM_D1 = 192, TM_O = 256, TM_S = 320, TM_COLS = 512;

__device__ __forceinline__ uint32_t tk_off(int r, int k) {
    return (uint32_t)((r >> 3) * 2048 + (k >> 2) * 128 + (r & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x rounded to tf32 (nearest, ties away from zero), kept in an fp32 word.
__device__ __forceinline__ float tf32r(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void st_op(uint8_t *sm, uint32_t base, int r, int k, float x) {
    *reinterpret_cast<float *>(sm + base + tk_off(r, k)) = tf32r(x);
}

// Instruction descriptor of kind::tf32 (fp32 accumulator, tf32 A and B, both K-major).
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                       // D format: f32
           | (2u << 7)                     // A format: tf32
           | (2u << 10)                    // B format: tf32
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void mma_tf32_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 q, %4, 0;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, q;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 q, %4, 0;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Descriptor of a K-major no-swizzle fp32 operand with 64 K-elements per row; one K step of the
// tf32 MMA (8 elements) is 2 core matrices, 256 bytes on.
__device__ __forceinline__ uint64_t opdesc(uint32_t saddr) { return sdesc(saddr, 128u, 2048u); }
constexpr uint64_t kStep = 256u >> 4;

template <bool GATED>
__global__ void __launch_bounds__(NT, 1) kda_prefill_tf32_kernel(const RunParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *gam = reinterpret_cast<float *>(sm + SM_GAM);
    float *cst = reinterpret_cast<float *>(sm + SM_CST);
    float *wsum = reinterpret_cast<float *>(sm + SM_WS);
    float *sbeta = reinterpret_cast<float *>(sm + SM_BETA);
    float *As = reinterpret_cast<float *>(sm + SM_AS);
    float *Xs = reinterpret_cast<float *>(sm + SM_X);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + SM_BAR);
    uint32_t *tptr = reinterpret_cast<uint32_t *>(sm + SM_TPTR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, d = p.dk;
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
    const float *qg = static_cast<const float *>(p.q), *kg = static_cast<const float *>(p.k);
    const float *vg = static_cast<const float *>(p.v), *gg = static_cast<const float *>(p.g);
    const float *bg = static_cast<const float *>(p.beta);
    float *og = static_cast<float *>(p.o);
    const size_t rs = (size_t)H * d;  // elements between consecutive tokens

    if (warp == 0) {
        tmem_alloc(tptr, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // V^T rows 64..127 (padded value columns) are zero for the whole run.
    for (int e = tid; e < 64 * 64; e += NT) st_op(sm, SM_VT, 64 + (e >> 6), e & 63, 0.f);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tptr, 0);
    const uint32_t sb = __shfl_sync(0xffffffffu, smem_u32(sm), 0);
    const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;  // TMEM lane quarter of warps 0..3

    // Initial state into TMEM: lane v holds S^T row v (column k = key channel); lanes >= d zero.
    if (warp < 4) {
        const int v = 32 * warp + lane;
        const long long init_off = p.init ? state_slot_offset(p.init_idx, p.pool, n, H, h, d, p.err) : -1;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            float buf[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int k = 32 * cb + i;
                buf[i] = (init_off >= 0 && v < d && k < d) ? p.init[init_off + (size_t)k * d + v] : 0.f;
            }
            tmem_st32(tmem + tq + TM_S + 32 * cb, buf);
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();

    uint32_t phase = 0;
    bool ok = true;
    // Issue-and-wait of a group of MMAs (warp 0 issues; every thread waits, bounded).
    // Every thread polls (test_wait: nothing else is left to run while the MMAs complete, and a
    // suspended try_wait resumes much later than a poll sees the phase change).
    auto poll = [&](uint32_t parity) -> bool {
        const uint64_t t0 = globaltimer();
        while (true) {
            uint32_t done;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(done)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
            if (done) return true;
            if (globaltimer() - t0 > kWaitNs) return false;
        }
    };
    auto mma_wait = [&]() -> bool {
        const bool w = poll(phase);
        phase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(w ? 1 : 0) != 0;
    };
    auto mma_done = [&]() -> bool {
        if (warp == 0) mma_commit_warp(bar);
        return mma_wait();
    };

    // Step 1 of chunk cc: Gam = cumsum of g per channel, the per-channel factors (into the buffer
    // of the chunk's parity) and beta. Chunk 0's runs before the loop, every later chunk's while
    // MMA1 of the chunk before it runs (Gam, beta and the block sums are free by then; the factors
    // of that chunk are still read after MMA1, hence two buffers).
    auto step1 = [&](int cc) {
        const long long q0 = bos + (long long)cc * C;
        const int ln = (int)min((long long)C, eos - q0);
        float *cs = cst + (cc & 1) * (CST_N * 64);
        const int ch = tid & 63, grp = tid >> 6;  // 4 groups of 16 rows
        float run = 0.f, loc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * grp + i;
            float x = 0.f;
            if (r < ln && ch < d) {
                x = gg[(size_t)(q0 + r) * rs + (size_t)h * d + ch];
                if (GATED) x = -p.gate_bound / (1.f + ex2f(-x * kLog2e));
            }
            run += x;
            loc[i] = run;
        }
        wsum[grp * 64 + ch] = run;
        if (tid < C) sbeta[tid] = tid < ln ? bg[(size_t)(q0 + tid) * H + h] : 0.f;
        __syncthreads();
        float add = 0.f;
        for (int gq = 0; gq < grp; ++gq) add += wsum[gq * 64 + ch];
#pragma unroll
        for (int i = 0; i < 16; ++i) gam[(16 * grp + i) * SG + ch] = loc[i] + add;
        __syncthreads();
        if (tid < 64) {
            const float G15 = gam[15 * SG + tid], G31 = gam[31 * SG + tid];
            const float G47 = gam[47 * SG + tid], G63 = gam[63 * SG + tid];
            cs[CST_M0 * 64 + tid] = G15 * kLog2e;
            cs[CST_M1 * 64 + tid] = G47 * kLog2e;
            cs[CST_C0 * 64 + tid] = ex2f((G31 - G15) * kLog2e);  // exp(Gam_31 - Gam_15)
            cs[CST_C1 * 64 + tid] = ex2f((G47 - G31) * kLog2e);  // exp(Gam_47 - Gam_31)
            cs[CST_GL * 64 + tid] = G63 * kLog2e;
            cs[CST_GAML * 64 + tid] = ex2f(G63 * kLog2e);
        }
        __syncthreads();
    };
    if (nchunks > 0) step1(0);

#pragma unroll 1
    for (int c = 0; c < nchunks && ok; ++c) {
        const long long r0 = bos + (long long)c * C;
        const int len = (int)min((long long)C, eos - r0);
        if (c + 1 < nchunks) {  // the next chunk's rows of q, k, v and g into L2 (thread = row, tensor)
            const long long rr = r0 + C + (tid & 63);
            if (rr < eos) {
                const int pt = tid >> 6;
                const float *a = (pt == 0 ? qg : pt == 1 ? kg : pt == 2 ? vg : gg) + (size_t)rr * rs + (size_t)h * d;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
                if (d > 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 32));
            }
        }

        const float *cs = cst + (c & 1) * (CST_N * 64);  // this chunk's per-channel factors

        // ---- 2. decay-scaled operands. Warp w owns rows 8w..8w+7: lane = row 8w + lane / 4 and
        // channels lane % 4 + 4i, so that the lanes of one store cover one 128-byte line of the
        // K-major core-matrix layout (and the rows' Gam entries fall in distinct banks).
        {
            const int r = 8 * warp + (lane >> 2), cq = lane & 3;
            const bool rlive = r < len;
            const int mh = r >> 5;
            const size_t e = (size_t)(r0 + r) * rs + (size_t)h * d;
            float kr[16], qr[16], vr[16];  // all of the thread's loads in flight at once
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int ch = 4 * i + cq;
                const bool live = rlive && ch < d;  // d is 32 or 64
                kr[i] = live ? kg[e + ch] : 0.f;
                qr[i] = live ? qg[e + ch] : 0.f;
                vr[i] = live ? vg[e + ch] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int ch = 4 * i + cq;
                const float kv = kr[i], qv = qr[i], vv = vr[i];
                const float G = gam[r * SG + ch] * kLog2e;
                // |Gam_r - ref| <= 80 for g in [-5, 0]; the clamps only keep factors finite
                const float ef = fminf(fmaxf(G - cs[(mh ? CST_M1 : CST_M0) * 64 + ch], -126.f), 126.f);
                const float f = ex2f(ef), fi = ex2f(-ef);
                st_op(sm, SM_APA, r, ch, kv * f);
                st_op(sm, SM_APA, 64 + r, ch, qv * f);
                st_op(sm, SM_APB, r, ch, kv * fi);
                if (mh) {  // off tile, A side: K and Q times exp(Gam_r - Gam_31)
                    const float c1 = cs[CST_C1 * 64 + ch];
                    st_op(sm, SM_OFFA, r - 32, ch, kv * f * c1);
                    st_op(sm, SM_OFFA, r, ch, qv * f * c1);
                } else {   // off tile, B side: K times exp(Gam_31 - Gam_r)
                    st_op(sm, SM_OFFB, r, ch, kv * fi * cs[CST_C0 * 64 + ch]);
                }
                const float fe = ex2f(fminf(G, 126.f));                                 // exp(Gam_r)
                const float fh = ex2f(fminf(cs[CST_GL * 64 + ch] - G, 126.f));         // exp(Gam_last - Gam_r)
                st_op(sm, SM_KQ, r, ch, kv * fe);
                st_op(sm, SM_KQ, 64 + r, ch, qv * fe);
                st_op(sm, SM_KHT, ch, r, kv * fh);
                st_op(sm, SM_VT, ch, r, vv);
            }
        }
        fence_async_smem();
        __syncthreads();

        // ---- 3. the A/P tiles -------------------------------------------------------------------
        if (warp == 0) {
            tc_fence_after();
            const uint64_t da = opdesc(sb + SM_APA), db = opdesc(sb + SM_APB);
            const uint64_t doa = opdesc(sb + SM_OFFA), dob = opdesc(sb + SM_OFFB);
#pragma unroll
            for (int st = 0; st < DP / 8; ++st)
                mma_tf32_warp(tmem + TM_AP, da + kStep * st, db + kStep * st, idesc_tf32(128, 64), st > 0);
#pragma unroll
            for (int st = 0; st < DP / 8; ++st)
                mma_tf32_warp(tmem + TM_OFF, doa + kStep * st, dob + kStep * st, idesc_tf32(64, 32), st > 0);
        }
        if (!(ok = mma_done())) break;

        // ---- 4. A and P out of TMEM (warps 0..3: lane quarter = warp) -----------------------------
        if (warp < 4) {
            float vals[32];
            const int L = 32 * warp + lane, i = L & 63;
            const int j0 = (warp & 1) ? 32 : 0;  // the diagonal half of row i
            tmem_ld32(tmem + tq + TM_AP + j0, vals);
            tmem_ld_wait();
            // 16-byte stores: a lane writes 4 consecutive entries of its row (A rows 272 bytes apart,
            // P rows in the core-matrix layout), 4 wavefronts per warp store.
            if (L < 64) {  // A row i (strictly lower, beta-scaled); the non-causal half is dropped by selection
                const float b = sbeta[i];
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4 *>(As + i * SA + j0 + k) =
                        make_float4((j0 + k < i) ? vals[k] * b : 0.f, (j0 + k + 1 < i) ? vals[k + 1] * b : 0.f,
                                    (j0 + k + 2 < i) ? vals[k + 2] * b : 0.f, (j0 + k + 3 < i) ? vals[k + 3] * b : 0.f);
                // rows 32..63, columns 0..31 come from the off tile below; rows 0..31, columns 32..63 are zero
                const int z0 = j0 == 32 ? 0 : 32;
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4 *>(As + i * SA + z0 + k) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {       // P row i (lower)
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4 *>(sm + SM_P + tk_off(i, j0 + k)) =
                        make_float4(tf32r((j0 + k <= i) ? vals[k] : 0.f), tf32r((j0 + k + 1 <= i) ? vals[k + 1] : 0.f),
                                    tf32r((j0 + k + 2 <= i) ? vals[k + 2] : 0.f), tf32r((j0 + k + 3 <= i) ? vals[k + 3] : 0.f));
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4 *>(sm + SM_P + tk_off(i, (32 - j0) + k)) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncthreads();  // the off tile overwrites part of the zeros above
        if (warp < 4) {
            float vals[32];
            tmem_ld32(tmem + tq + TM_OFF, vals);
            tmem_ld_wait();
            if (lane < 16) {  // off tile (M = 64): rows in lanes 0..15 of each quarter
                const int i = 32 + 16 * (warp & 1) + lane;
                if (warp < 2) {
                    const float b = sbeta[i];
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(As + i * SA + k) =
                            make_float4(vals[k] * b, vals[k + 1] * b, vals[k + 2] * b, vals[k + 3] * b);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(sm + SM_P + tk_off(i, k)) =
                            make_float4(tf32r(vals[k]), tf32r(vals[k + 1]), tf32r(vals[k + 2]), tf32r(vals[k + 3]));
                }
            }
        }
        __syncthreads();

        // ---- 5. X = (I + A)^{-1} in blocks: the four 16 x 16 diagonal blocks by forward
        // substitution (thread = one column of one block), then the 16 -> 32 and 32 -> 64 merges
        // X_BA = -X_BB (A_BA X_AA) as fp32 products on the CUDA cores; T = X Diag(beta). The
        // scratch of the merges is the Gam buffer (read by nothing after the operand build).
        {
            float *Ys = gam;
            for (int e = tid; e < 64 * 64; e += NT) Xs[(e >> 6) * SA + (e & 63)] = 0.f;
            __syncthreads();
            if (tid < 64) {  // column jj of diagonal block B0, held in registers (entries above jj are 0)
                const int B0 = 16 * (tid >> 4), jj = tid & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc = 0.f;  // the terms k < jj are A x 0 and leave acc at +0
#pragma unroll
                    for (int k = 0; k < i; ++k) acc = fmaf(As[(B0 + i) * SA + B0 + k], x[k], acc);
                    x[i] = i < jj ? 0.f : (i == jj ? 1.f : -acc);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) Xs[(B0 + i) * SA + B0 + jj] = x[i];
            }
            __syncthreads();
            // Each thread: one row x 4 consecutive columns of a product (one left entry and one
            // 16-byte right vector per K step), every entry summed in K order.
            auto fma4 = [](float (&acc)[4], float a, float4 x) {
                acc[0] = fmaf(a, x.x, acc[0]); acc[1] = fmaf(a, x.y, acc[1]);
                acc[2] = fmaf(a, x.z, acc[2]); acc[3] = fmaf(a, x.w, acc[3]);
            };
            if (tid < 128) {  // 16 -> 32, blocks (1, 0) and (3, 2): Y = A_IJ X_JJ
                const int pp = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
                const int I = 2 * pp + 1, J = 2 * pp;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    fma4(acc, As[(16 * I + r) * SA + 16 * J + k],
                         *reinterpret_cast<const float4 *>(Xs + (16 * J + k) * SA + 16 * J + c4));
                *reinterpret_cast<float4 *>(Ys + pp * 256 + r * 16 + c4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            }
            __syncthreads();
            if (tid < 128) {  // X_IJ = -X_II Y
                const int pp = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
                const int I = 2 * pp + 1, J = 2 * pp;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    fma4(acc, Xs[(16 * I + r) * SA + 16 * I + k], *reinterpret_cast<const float4 *>(Ys + pp * 256 + k * 16 + c4));
                *reinterpret_cast<float4 *>(Xs + (16 * I + r) * SA + 16 * J + c4) = make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
            }
            __syncthreads();
            {  // 32 -> 64: Y = A_BA X_AA
                const int r = tid >> 3, c4 = 4 * (tid & 7);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int k = 0; k < 32; ++k)
                    fma4(acc, As[(32 + r) * SA + k], *reinterpret_cast<const float4 *>(Xs + k * SA + c4));
                *reinterpret_cast<float4 *>(Ys + r * 32 + c4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            }
            __syncthreads();
            {  // X_BA = -X_BB Y
                const int r = tid >> 3, c4 = 4 * (tid & 7);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int k = 0; k < 32; ++k)
                    fma4(acc, Xs[(32 + r) * SA + 32 + k], *reinterpret_cast<const float4 *>(Ys + k * 32 + c4));
                *reinterpret_cast<float4 *>(Xs + (32 + r) * SA + c4) = make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
            }
            __syncthreads();
            // T = X Diag(beta), 16 bytes per lane: rows 8 w + lane % 8 (one 128-byte line of the
            // core-matrix layout per 8 lanes), columns 16 q + 4 (lane / 8) .. + 3.
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = 8 * warp + (lane & 7), jc = 16 * q + 4 * (lane >> 3);
                const float4 x = *reinterpret_cast<const float4 *>(Xs + i * SA + jc);
                const float4 b = *reinterpret_cast<const float4 *>(sbeta + jc);
                *reinterpret_cast<float4 *>(sm + SM_T + tk_off(i, jc)) =
                    make_float4(tf32r(x.x * b.x), tf32r(x.y * b.y), tf32r(x.z * b.z), tf32r(x.w * b.w));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 6. MMA1: [K+ S | Q+ S]^T = S^T [K+ ; Q+]^T (the fp32 state in TMEM as the A operand) --
        if (warp == 0) {
            tc_fence_after();
            const uint64_t dkq = opdesc(sb + SM_KQ);
#pragma unroll
            for (int st = 0; st < DP / 8; ++st)
                mma_tf32_tmem_a_warp(tmem + TM_D1, tmem + TM_S + 8 * st, dkq + kStep * st, idesc_tf32(128, 128),
                                     st > 0);
            mma_commit_warp(bar);
        }
        if (c + 1 < nchunks) step1(c + 1);  // step 1 of the next chunk while MMA1 runs
        if (!(ok = mma_wait())) break;

        // ---- 7. -(K+ S)^T as MMA2's second A operand; S <- S Diag(gam_last) ---------------------
        if (warp < 4) {
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float x[32];
                tmem_ld32(tmem + tq + TM_D1 + 32 * cb, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = -x[i];
                tmem_st32(tmem + tq + TM_RA + 32 * cb, x);
                tmem_ld32(tmem + tq + TM_S + 32 * cb, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] *= cs[CST_GAML * 64 + 32 * cb + i];
                tmem_st32(tmem + tq + TM_S + 32 * cb, x);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();

        // ---- 8. MMA2: U^T = V^T T^T - (K+ S)^T T^T (into the columns of K+ S) --------------------
        if (warp == 0) {
            tc_fence_after();
            const uint64_t dv = opdesc(sb + SM_VT), dt = opdesc(sb + SM_T);
#pragma unroll
            for (int st = 0; st < C / 8; ++st)
                mma_tf32_warp(tmem + TM_D1, dv + kStep * st, dt + kStep * st, idesc_tf32(128, 64), st > 0);
#pragma unroll
            for (int st = 0; st < C / 8; ++st)
                mma_tf32_tmem_a_warp(tmem + TM_D1, tmem + TM_RA + 8 * st, dt + kStep * st, idesc_tf32(128, 64), 1u);
        }
        if (!(ok = mma_done())) break;

        // ---- 9. U^T as the A operand of MMA3 and MMA4 --------------------------------------------
        if (warp < 4) {
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float x[32];
                tmem_ld32(tmem + tq + TM_D1 + 32 * cb, x);
                tmem_ld_wait();
                tmem_st32(tmem + tq + TM_RA + 32 * cb, x);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();

        // ---- 10. MMA3: O^T += U^T P^T (onto (Q+ S)^T); MMA4: S^T += U^T Khat ---------------------
        if (warp == 0) {
            tc_fence_after();
            const uint64_t dp = opdesc(sb + SM_P), dkh = opdesc(sb + SM_KHT);
#pragma unroll
            for (int st = 0; st < C / 8; ++st)
                mma_tf32_tmem_a_warp(tmem + TM_O, tmem + TM_RA + 8 * st, dp + kStep * st, idesc_tf32(128, 64), 1u);
#pragma unroll
            for (int st = 0; st < C / 8; ++st)
                mma_tf32_tmem_a_warp(tmem + TM_S, tmem + TM_RA + 8 * st, dkh + kStep * st, idesc_tf32(128, 64), 1u);
        }
        if (!(ok = mma_done())) break;

        // ---- 11. O out: O^T (lane = value column) into a [token][value] staging tile in the A/P
        // operand region (free until the next chunk's build), then every thread stores rows of it.
        {
            float *Ost = reinterpret_cast<float *>(sm + SM_APA);  // [64 tokens][SA]
            if (warp < 2) {
                const int v = 32 * warp + lane;
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    float x[32];
                    tmem_ld32(tmem + tq + TM_O + 32 * cb, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) Ost[(32 * cb + i) * SA + v] = x[i];
                }
            }
            __syncthreads();
            const int v = tid & 63;
#pragma unroll 4
            for (int t = tid >> 6; t < 64; t += 4)
                if (t < len && v < d) og[(size_t)(r0 + t) * rs + (size_t)h * d + v] = Ost[t * SA + v];
        }
        tc_fence_before();
        __syncthreads();  // the next chunk's operands overwrite what these MMAs read
    }

    if (ok) {
        const long long fin_off = p.fin ? state_slot_offset(p.fin_idx, p.pool, n, H, h, d, p.err) : -1;
        if (fin_off >= 0 && warp < 2) {
            const int v = 32 * warp + lane;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float x[32];
                tmem_ld32(tmem + tq + TM_S + 32 * cb, x);
                tmem_ld_wait();
                if (v < d)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (32 * cb + i < d) p.fin[fin_off + (size_t)(32 * cb + i) * d + v] = x[i];
            }
        }
    } else if (tid == 0) {
        atomicOr(p.err, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

// fp32 with d_k == d_v in {32, 64}, without the L2 normalisation and the output gate (those run
// on the CUDA-core recurrence).
bool tf32_prefill_supported(kda_dtype dtype, int dk, int dv, const RunParams &p) {
    return dtype == KDA_F32 && dk == dv && (dk == 32 || dk == 64) && !p.qk_l2norm && !p.out_gate && !p.dump;
}

cudaError_t launch_tf32_prefill(const RunParams &p, cudaStream_t s) {
    static std::mutex mu;
    static bool attr_set[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute((const void *)kda_prefill_tf32_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute((const void *)kda_prefill_tf32_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const void *fn = p.gate_bound > 0.f ? (const void *)kda_prefill_tf32_kernel<true>
                                        : (const void *)kda_prefill_tf32_kernel<false>;
    void *args[] = {(void *)&p};
    return cudaLaunchKernel(fn, dim3((unsigned)(p.n_seqs * p.H)), dim3(NT), args, SMEM_BYTES, s);
}

}  // namespace kda
