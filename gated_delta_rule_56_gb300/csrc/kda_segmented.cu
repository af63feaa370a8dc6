// kda_segmented.cu -- prefill of a few long sequences, split along the sequence so that more
// CTAs than (sequence, head) pairs share the work.
//
// The recurrence of "Kimi Delta Attention: the linear core" (maidul-haque blog) is affine in the
// state (its per-token transition does not depend on it): over a segment p of a sequence, S_t = M_{p,t} S_start + S^loc_t, where S^loc_t is the
// state reached from zero and M_{p,t} the product of the segment's per-token transitions
// (I - beta k k^T) Diag(exp g) up to t. The read-out is then
//     o_t = S_t^T q_t = (S^loc_t)^T q_t + S_start^T (M_{p,t}^T q_t) = o^loc_t + S_start^T qt_t.
// Both parts come from the chunked tensor-core kernel run over the segments as independent
// sequences: from a zero state (o^loc, S^loc at the segment end), and with v = 0 from the identity
// (its read-out is qt_t = M_{p,t}^T q_t, its final state the segment transition M_p). Then
//     S_start of segment 0 = the initial state,  S_start of p + 1 = M_p S_start(p) + S^loc(p)
// (a short scan per (sequence, head), which also gives the final state), and one GEMM per tile
// of tokens adds S_start^T qt_t to o^loc. Exact up to rounding; at most twice the work of one
// pass, spread over P times as many CTAs.
//
// The transition run first covers only the first kHorizon rows of every segment. With v = 0 a
// state that is exactly zero stays exactly zero (every later MMA multiplies zeros), so where M is
// all zeros after the horizon, every later qt_t and the segment transition are exactly zero and
// the rest of the run is skipped. Only the (segment, head) pairs whose M is not yet zero (slowly
// decaying gates) run the whole segment again.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int D = 128;                      // d_k == d_v
constexpr int CT = 128;                     // tokens per correction tile
constexpr int kMinSegRows = 32 * 64;        // segments of at least 32 chunks
constexpr int kMaxSegments = 8;
constexpr int kHorizon = 4 * 64;            // rows of the first transition run
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait

struct Plan {
    int P = 0;        // segments per sequence
    int Ls = 0;       // rows per segment (the last one may be shorter)
    size_t off_cu = 0, off_qt = 0, off_sloc = 0, off_mtr = 0, off_sst = 0, off_done = 0, bytes = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Segment count and workspace layout on a GPU with `sms` SMs, or P == 0 when a single pass is
// the better choice.
Plan make_plan_for(int B, int T, int H, int sms) {
    Plan pl;
    if (sms <= 0) return pl;
    const long long pairs = (long long)B * H;
    if (pairs <= 0 || T <= 0) return pl;
    // One wave: as many segments as fit next to each other on the SMs. (A split into several
    // waves with every SM busy, e.g. 19 segments = 608 CTAs = 4 waves for 32 heads, ran each
    // chunk about 24 % slower: the kernel's aggregate rate stays near the same total when more
    // SMs run it, so more, shorter segments do not pay for the extra passes.)
    const long long P = std::min<long long>(std::min<long long>(kMaxSegments, sms / pairs), T / kMinSegRows);
    if (P < 2) return pl;
    const long long per = (T + P - 1) / P;
    pl.Ls = (int)((per + 63) / 64 * 64);
    pl.P = (int)((T + pl.Ls - 1) / pl.Ls);
    const long long segs = (long long)B * pl.P;
    size_t off = 0;
    pl.off_cu = off;
    off = align256(off + (size_t)(segs + 1) * 4);
    pl.off_qt = off;
    off = align256(off + (size_t)B * T * H * D * 2);
    pl.off_sloc = off;
    off = align256(off + (size_t)segs * H * D * D * 4);
    pl.off_mtr = off;
    off = align256(off + (size_t)segs * H * D * D * 4);
    pl.off_sst = off;
    off = align256(off + (size_t)segs * H * D * D * 2);
    pl.off_done = off;
    off = align256(off + (size_t)segs * H);
    pl.bytes = off;
    return pl;
}

// The plan for the current device.
Plan make_plan(int B, int T, int H) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return Plan{};
    return make_plan_for(B, T, H, sms);
}

// cu_seqlens of the segments as packed sequences: segment p of sequence b covers rows
// b*T + p*Ls .. b*T + min((p+1)*Ls, T) - 1.
__global__ void seg_bounds_kernel(int32_t *cu, int B, int T, int P, int Ls) {
    const int n = B * P;
    for (int i = threadIdx.x; i <= n; i += blockDim.x) {
        if (i == n) {
            cu[i] = B * T;
        } else {
            const int b = i / P, p = i % P;
            cu[i] = b * T + p * Ls;
        }
    }
}

// done[i] = 1 when the transition of (segment, head) i after the horizon is exactly zero (nothing
// further to compute) or the pair was not run (skip[i]), else 0. One CTA of 256 threads per pair.
__global__ void __launch_bounds__(256) seg_done_kernel(const float *__restrict__ mtr, const uint8_t *__restrict__ skip,
                                                       uint8_t *__restrict__ done) {
    if (skip && skip[blockIdx.x]) {
        if (threadIdx.x == 0) done[blockIdx.x] = 1;
        return;
    }
    const float4 *m = reinterpret_cast<const float4 *>(mtr + (size_t)blockIdx.x * D * D);
    bool zero = true;
    for (int e = threadIdx.x; e < D * D / 4; e += 256) {
        const float4 x = m[e];
        zero = zero && x.x == 0.f && x.y == 0.f && x.z == 0.f && x.w == 0.f;
    }
    zero = __syncthreads_and(zero) != 0;
    if (threadIdx.x == 0) done[blockIdx.x] = zero ? 1 : 0;
}

// One CTA per (sequence b, head h). Equal segments (seg_first == NULL: segments b*P .. b*P+P-1, all
// run from a zero state): S_start(0) = init (or 0), S_start(p+1) = M_p S_start(p) + S^loc(p).
// Planned segments of packed sequences (seg_first != NULL: segments seg_first[b] .. seg_first[b+1]-1,
// the first one run from the sequence's initial state, so that its S^loc is already the state at
// its end): S_start(first + 1) = S^loc(first), and the same recursion after it.
// S_start(p) is stored transposed in bf16 (the B operand of the correction GEMM), and the state
// after the last segment is the final state. Thread (ti, tj) owns the 8 x 8 block at (8 ti, 8 tj).
__global__ void __launch_bounds__(256) seg_scan_kernel(const float *__restrict__ mtr, const float *__restrict__ sloc,
                                                       const float *__restrict__ init, float *__restrict__ fin,
                                                       const int32_t *init_idx, const int32_t *fin_idx, int pool,
                                                       unsigned *err, __nv_bfloat16 *__restrict__ sst, int P, int H,
                                                       const int32_t *__restrict__ seg_first) {
    extern __shared__ float S[];  // [128][132]
    constexpr int LD = 132;
    const int bh = blockIdx.x, b = bh / H, h = bh % H, tid = threadIdx.x;
    const int ti = tid >> 4, tj = tid & 15;
    const long long fin_off = fin ? state_slot_offset(fin_idx, pool, b, H, h, D, err) : -1;
    int s_begin, s_end;
    if (seg_first) {
        const int s0 = seg_first[b];
        s_begin = s0 + 1;
        s_end = max(seg_first[b + 1], s_begin);
        const float *L0 = sloc + ((size_t)s0 * H + h) * D * D;
        for (int e = tid; e < D * D; e += 256) S[(e >> 7) * LD + (e & 127)] = L0[e];
    } else {
        s_begin = b * P;
        s_end = s_begin + P;
        const long long init_off = init ? state_slot_offset(init_idx, pool, b, H, h, D, err) : -1;
        for (int e = tid; e < D * D; e += 256)
            S[(e >> 7) * LD + (e & 127)] = init_off >= 0 ? init[init_off + e] : 0.f;
    }
    __syncthreads();
#pragma unroll 1
    for (int sg = s_begin; sg < s_end; ++sg) {
        const size_t s = (size_t)sg * H + h;
        for (int e = tid; e < D * D; e += 256) {  // S_start^T: row v, column k
            const int v = e >> 7, k = e & 127;
            sst[s * D * D + e] = __float2bfloat16_rn(S[k * LD + v]);
        }
        const float *M = mtr + s * D * D, *L = sloc + s * D * D;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = L[(8 * ti + i) * D + 8 * tj + j];
#pragma unroll 2
        for (int k = 0; k < D; ++k) {
            float a[8], c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = M[(8 * ti + i) * D + k];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = S[k * LD + 8 * tj + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], c[j], acc[i][j]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) S[(8 * ti + i) * LD + 8 * tj + j] = acc[i][j];
        __syncthreads();
    }
    if (fin_off >= 0)
        for (int e = tid; e < D * D; e += 256) fin[fin_off + e] = S[(e >> 7) * LD + (e & 127)];
}

// Offset of the 16-byte chunk (row r, channels 8j..8j+7) of an R-row operand in the
// 128-byte-swizzled K-major layout (the layout of the TMA tiles).
__device__ __forceinline__ uint32_t sw_chunk(int r, int j, int R) {
    return (uint32_t)((j >> 3) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 + (((j & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t ksw(int st, uint32_t rows) {
    return (uint64_t)(((uint32_t)(st >> 2) * rows * 128u + (uint32_t)(st & 3) * 32u) >> 4);
}

// max |x| over a block of 128 threads; a NaN anywhere makes the result NaN.
__device__ __forceinline__ float block_absmax(float m, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float t = __shfl_xor_sync(0xffffffffu, m, o);
        m = (t > m || t != t) ? t : m;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < 4; ++w) r = (red[w] > r || red[w] != red[w]) ? red[w] : r;
    return r;
}

__device__ __forceinline__ float absmax_bf16x8(const uint4 w, float m) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo = fabsf(__uint_as_float(ww[e] << 16)), hi = fabsf(__uint_as_float(ww[e] & 0xffff0000u));
        m = (lo > m || lo != lo) ? lo : m;
        m = (hi > m || hi != hi) ? hi : m;
    }
    return m;
}

// o[t] += S_start^T qt[t] over the tiles of 128 tokens of segment blockIdx.y and head blockIdx.z, CTA
// x taking tiles x, x + gridDim.x, ...: per tile D = qt_tile (128 x 128) x S_start (128 x 128) on the
// tensor core (A: the qt tile by TMA, B: S_start^T, loaded once), then o read, added and written back
// row by row (thread = token). A tile whose correction is bounded by 128 max|S_start| max|qt| < 1e-30
// is left as it is (qt decays with the segment transition; such a term cannot change a bf16 output).
// Segment geometry: equal segments (seg_cu == NULL): segment b * P + p covers rows p*Ls .. of batch
// row b (T rows each), and segments p < p0 are skipped (zero S_start); planned segments of packed
// sequences (seg_cu != NULL): rows seg_cu[s] .. seg_cu[s+1]-1, and the first segment of a sequence
// (is_first[s]) needs no correction.
constexpr int kTilesPerCta = 8;
constexpr float kNegligible = 1e-30f;

__global__ void __launch_bounds__(128) seg_correct_kernel(const __grid_constant__ CUtensorMap qt_map,
                                                          const __nv_bfloat16 *__restrict__ sst,
                                                          const uint8_t *__restrict__ done,
                                                          __nv_bfloat16 *__restrict__ o,
                                                          const __nv_bfloat16 *__restrict__ zg, int T, int H, int Ls,
                                                          int P, int p0, const int32_t *__restrict__ seg_cu,
                                                          const uint8_t *__restrict__ is_first, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = sm, *sB = sm + 32768;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + 65536);
    uint32_t *tptr = reinterpret_cast<uint32_t *>(sm + 65536 + 16);
    float *red = reinterpret_cast<float *>(sm + 65536 + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.y, h = blockIdx.z;
    long long base, len;  // packed row of the segment start, and its rows
    if (seg_cu) {
        if (is_first[seg]) return;
        base = seg_cu[seg];
        len = (long long)seg_cu[seg + 1] - base;
    } else {
        const int b = seg / P, p = seg % P;
        if (p < p0) return;  // S_start is zero: nothing to add
        base = (long long)b * T + (long long)p * Ls;
        len = min((long long)Ls, (long long)T - (long long)p * Ls);
    }
    // qt is exactly zero past the horizon where the transition run stopped early (and not stored).
    const long long hi = min(len, done[(size_t)seg * H + h] ? (long long)kHorizon : len);
    if ((long long)blockIdx.x * CT >= hi) return;

    if (warp == 0) {
        tmem_alloc(tptr, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    const __nv_bfloat16 *src = sst + ((size_t)seg * H + h) * D * D;
    float smax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int idx = tid + 128 * i, r = idx >> 4, j = idx & 15;
        const uint4 w = *reinterpret_cast<const uint4 *>(src + r * D + 8 * j);
        smax = absmax_bf16x8(w, smax);
        *reinterpret_cast<uint4 *>(sB + sw_chunk(r, j, 128)) = w;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tptr;
    smax = block_absmax(smax, red);

    bool ok = true;
    uint32_t ncopy = 0, nmma = 0;  // copies and MMA groups issued (their barrier phases)
    const uint64_t da = sdesc_sw128(smem_u32(sA), 16u, 1024u), db = sdesc_sw128(smem_u32(sB), 16u, 1024u);
#pragma unroll 1
    for (long long r0 = (long long)blockIdx.x * CT; r0 < hi && ok; r0 += (long long)gridDim.x * CT) {
        const int nrows = (int)min((long long)CT, hi - r0);
        const long long row = base + r0;  // packed row of the tile start
        if (tid == 0) {
            mbar_arrive_expect_tx(&bars[0], 32768);
            for (int rb = 0; rb < 2; ++rb)
                for (int cb = 0; cb < 2; ++cb)  // rows past the tensor read as 0; past the segment are not stored
                    tma_load_3d(sA + cb * 16384 + rb * 8192, &qt_map, &bars[0], 64 * cb, h, (int)(row + 64 * rb));
        }
        ok = __syncthreads_and(mbar_wait(&bars[0], ncopy & 1u, kWaitNs)) != 0;
        ++ncopy;
        if (!ok) break;
        float qmax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) qmax = absmax_bf16x8(*reinterpret_cast<const uint4 *>(sA + 16 * (tid + 128 * i)), qmax);
        qmax = block_absmax(qmax, red);
        if (qmax * smax * 128.f < kNegligible) {  // false for NaN: a NaN is always propagated
            __syncthreads();                      // everyone has read sA before the next copy
            continue;
        }
        if (warp == 0) {
            tc_fence_after();
#pragma unroll
            for (int st = 0; st < D / 16; ++st)
                mma_bf16_warp(tmem, da + ksw(st, 128), db + ksw(st, 128), idesc_bf16(128, 128), st > 0);
            mma_commit_warp(&bars[1]);
        }
        ok = __syncthreads_and(mbar_wait(&bars[1], nmma & 1u, kWaitNs)) != 0;
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        const int rl = 32 * warp + lane;  // tile row = TMEM lane
        __nv_bfloat16 *orow = o + ((size_t)(row + rl) * H + h) * D;
        // With an output gate the local pass stored sigmoid(z) o_loc, so the correction adds sigmoid(z) S^T qt.
        const __nv_bfloat16 *zrow = zg ? zg + ((size_t)(row + rl) * H + h) * D : nullptr;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            float acc[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * cb, acc);
            tmem_ld_wait();
            if (rl < nrows) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w = *reinterpret_cast<const uint4 *>(orow + 32 * cb + 8 * q);
                    uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                    if (zrow) {
                        const uint4 z = __ldg(reinterpret_cast<const uint4 *>(zrow + 32 * cb + 8 * q));
                        const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[8 * q + 2 * e] *= __fdividef(1.f, 1.f + __expf(-__uint_as_float(zw[e] << 16)));
                            acc[8 * q + 2 * e + 1] *= __fdividef(1.f, 1.f + __expf(-__uint_as_float(zw[e] & 0xffff0000u)));
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo_v = __uint_as_float(ww[e] << 16) + acc[8 * q + 2 * e];
                        const float hi_v = __uint_as_float(ww[e] & 0xffff0000u) + acc[8 * q + 2 * e + 1];
                        ww[e] = pack_bf16(lo_v, hi_v);
                    }
                    *reinterpret_cast<uint4 *>(orow + 32 * cb + 8 * q) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // TMEM read out and sA consumed before the next tile
        tc_fence_after();
    }
    if (!ok && tid == 0) {  // a wait ran out: record it, and leave nothing in flight (bounded)
        atomicOr(err, kErrTimeout);
        (void)mbar_wait(&bars[0], (ncopy - 1) & 1u, kWaitNs);
        if (nmma) (void)mbar_wait(&bars[1], (nmma - 1) & 1u, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// Segments of one packed sequence of L rows for a target segment length: P equal segments of Ls
// rows (whole chunks; the last one shorter), at most kMaxSegments. The same arithmetic on the host
// (a single packed sequence, whose length is the packed rows) and in the planner kernel.
__host__ __device__ inline void packed_segments_of(long long L, long long target, long long &P, long long &Ls) {
    P = L <= 0 ? 1 : (L + target - 1) / target;
    if (P > kMaxSegments) P = kMaxSegments;
    if (P < 1) P = 1;
    Ls = ((L + P - 1) / P + 63) / 64 * 64;
    if (Ls < 64) Ls = 64;
    P = L <= 0 ? 1 : (L + Ls - 1) / Ls;
}

__host__ __device__ inline long long packed_target_rows(int T, int slots) {
    const long long per = ((long long)T + slots - 1) / slots;
    const long long t = (per + 63) / 64 * 64;
    return t > kMinSegRows ? t : (long long)kMinSegRows;
}

// Plan of the split of packed sequences, made on the device from cu_seqlens (one CTA). With
// `slots` = SMs / H CTAs per head to fill, the target segment length is the packed rows / slots
// (rounded up to whole chunks, at least kMinSegRows), and sequence n gets P_n = min(kMaxSegments,
// ceil(L_n / target)) segments of equal length (whole chunks; the last one shorter). Outputs, for
// S_max planned segments (those past the S used are empty, at row T, and skipped): seg_cu[S_max + 1]
// (bounds as packed rows), seg_first[n + 1] (first segment of each sequence, then S), seg_init[S_max]
// (the state slot a segment starts from: the sequence's initial state for its first segment, none for
// the others), is_first[S_max] and skip[S_max * H] (pairs the transition run leaves out: first and
// empty segments). A cu_seqlens that does not start at 0, decreases or does not end at T is reported
// (kErrBadSeqlens) and planned as clamped bounds, one segment per sequence.
__global__ void __launch_bounds__(256) seg_plan_packed_kernel(const int32_t *__restrict__ cu, int n, int T, int H,
                                                              int slots, int S_max, const int32_t *__restrict__ init_idx,
                                                              int32_t *__restrict__ seg_cu, int32_t *__restrict__ seg_first,
                                                              int32_t *__restrict__ seg_init, uint8_t *__restrict__ is_first,
                                                              uint8_t *__restrict__ skip, unsigned *err) {
    __shared__ int used;
    if (threadIdx.x == 0) {
        bool bad = cu[0] != 0 || cu[n] != T;
        for (int i = 0; i < n && !bad; ++i) bad = cu[i + 1] < cu[i];
        if (bad) atomicOr(err, kErrBadSeqlens);
        const long long target = packed_target_rows(T, slots);
        int sg = 0;
        long long prev = 0;
        for (int i = 0; i < n; ++i) {
            long long b0 = bad ? min(max(prev, (long long)cu[i]), (long long)T) : cu[i];
            long long b1 = bad ? min(max(b0, (long long)cu[i + 1]), (long long)T) : cu[i + 1];
            prev = b1;
            const long long L = b1 - b0;
            long long P, Ls;
            packed_segments_of(L, target, P, Ls);
            if (bad) {
                P = 1;
                Ls = L > 64 ? L : 64;
            }
            seg_first[i] = sg;
            for (int q = 0; q < P && sg < S_max; ++q, ++sg) {
                seg_cu[sg] = (int32_t)min(b0 + q * Ls, b1);
                seg_init[sg] = q == 0 ? (init_idx ? init_idx[i] : i) : -1;
                is_first[sg] = q == 0 ? 1 : 0;
            }
        }
        seg_first[n] = sg;
        used = sg;
        for (int q = sg; q <= S_max; ++q) {
            seg_cu[q] = T;
            if (q < S_max) {
                seg_init[q] = -1;
                is_first[q] = 1;
            }
        }
    }
    __syncthreads();
    const int S = used;
    for (int e = threadIdx.x; e < S_max * H; e += blockDim.x) {
        const int q = e / H;
        skip[e] = (q >= S || is_first[q] || seg_cu[q + 1] == seg_cu[q]) ? 1 : 0;
    }
}

// Workspace layout of the packed split; bytes == 0 when such a call is not split.
struct PackedPlan {
    int slots = 0, S_max = 0;
    size_t off_cu = 0, off_first = 0, off_init = 0, off_isfirst = 0, off_skip = 0, off_qt = 0, off_sloc = 0,
           off_mtr = 0, off_sst = 0, off_done = 0, bytes = 0;
};

PackedPlan make_packed_plan_for(int n, int T, int H, int sms) {
    PackedPlan pl;
    if (sms <= 0 || n <= 0 || H <= 0 || T < 2 * kMinSegRows) return pl;
    const int slots = sms / H;
    if (slots < 2 || n >= slots) return pl;  // as many sequences as CTAs per head: nothing to gain
    pl.slots = slots;
    // A bound on the planned segments (each sequence gets at most ceil(L_n / target) <= L_n / target + 1
    // of them, and the targets add up to at most `slots`). Blocks of unused segments are launched and
    // exit at once, but they change how the hardware places the others (measured: a quarter more
    // blocks than segments made the pass 20 % slower), so a single sequence -- its length is the
    // packed rows -- is planned exactly here.
    if (n == 1) {
        long long P, Ls;
        packed_segments_of(T, packed_target_rows(T, slots), P, Ls);
        if (P < 2) return PackedPlan{};
        pl.S_max = (int)P;
    } else {
        pl.S_max = (int)std::min<long long>((long long)kMaxSegments * n, (long long)n + slots);
    }
    const long long S = pl.S_max;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    pl.off_cu = take((size_t)(S + 1) * 4);
    pl.off_first = take((size_t)(n + 1) * 4);
    pl.off_init = take((size_t)S * 4);
    pl.off_isfirst = take((size_t)S);
    pl.off_skip = take((size_t)S * H);
    pl.off_qt = take((size_t)T * H * D * 2);
    pl.off_sloc = take((size_t)S * H * D * D * 4);
    pl.off_mtr = take((size_t)S * H * D * D * 4);
    pl.off_sst = take((size_t)S * H * D * D * 2);
    pl.off_done = take((size_t)S * H);
    pl.bytes = off;
    return pl;
}

PackedPlan make_packed_plan(int n, int T, int H) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PackedPlan{};
    return make_packed_plan_for(n, T, H, sms);
}

constexpr int kScanSmem = 128 * 132 * 4;
constexpr int kCorrectSmem = 65536 + 64 + 1024;  // A, B, barriers, TMEM address, block max

// Shared-memory limits of the scan and correction kernels, once per device.
cudaError_t set_segmented_attributes() {
    static std::mutex mu;
    static bool attr_set[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(seg_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCorrectSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace

void segmented_plan_for(int B, int T, int H, int sms, int *P, int *Ls, size_t *bytes) {
    const Plan pl = (long long)B * T >= 0x7fffffffLL - 64 ? Plan{} : make_plan_for(B, T, H, sms);
    *P = pl.P;
    *Ls = pl.Ls;
    *bytes = pl.bytes;
}

size_t segmented_workspace_bytes(kda_dtype dtype, int B, int T, int H, int dk, int dv, bool varlen) {
    if (dtype != KDA_BF16 || dk != D || dv != D || varlen) return 0;
    if ((long long)B * T >= 0x7fffffffLL - 64) return 0;
    return make_plan(B, T, H).bytes;
}

size_t segmented_packed_workspace_bytes_for(kda_dtype dtype, int n_seqs, int T, int H, int dk, int dv, int sms) {
    if (dtype != KDA_BF16 || dk != D || dv != D || T >= 0x7fffffff - 64) return 0;
    return make_packed_plan_for(n_seqs, T, H, sms).bytes;
}

cudaError_t launch_segmented_packed_prefill(const RunParams &p, void *workspace, size_t workspace_bytes,
                                            cudaStream_t s) {
    const int T = p.T, H = p.H, n = p.n_seqs;
    const PackedPlan pl = make_packed_plan(n, T, H);
    if (!pl.bytes || workspace_bytes < pl.bytes || !workspace) return cudaErrorInvalidValue;
    cudaError_t e = set_segmented_attributes();
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *seg_cu = reinterpret_cast<int32_t *>(ws + pl.off_cu);
    int32_t *seg_first = reinterpret_cast<int32_t *>(ws + pl.off_first);
    int32_t *seg_init = reinterpret_cast<int32_t *>(ws + pl.off_init);
    uint8_t *is_first = ws + pl.off_isfirst;
    uint8_t *skip = ws + pl.off_skip;
    __nv_bfloat16 *qt = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_qt);
    float *sloc = reinterpret_cast<float *>(ws + pl.off_sloc);
    float *mtr = reinterpret_cast<float *>(ws + pl.off_mtr);
    __nv_bfloat16 *sst = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_sst);
    uint8_t *done = ws + pl.off_done;
    const int S = pl.S_max;

    seg_plan_packed_kernel<<<1, 256, 0, s>>>(p.cu_seqlens, n, T, H, pl.slots, S, p.init_idx, seg_cu, seg_first,
                                             seg_init, is_first, skip, p.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // Pass 1: every segment; the first one of a sequence from its initial state (its end state is
    // then that of the sequence), the others from zero (o^loc into o, S^loc into the workspace).
    RunParams pa = p;
    pa.cu_seqlens = seg_cu;
    pa.n_seqs = S;
    pa.init_idx = p.init ? seg_init : nullptr;
    pa.pool = p.init_idx ? p.pool : n;
    pa.fin = sloc;
    pa.fin_idx = nullptr;
    pa.order = nullptr;
    pa.zero_v = false;
    pa.identity_init = false;
    pa.max_chunks = 0;
    pa.skip = nullptr;
    if ((e = launch_tc_prefill(pa, s)) != cudaSuccess) return e;
    // Pass 2: v = 0 from the identity for the later segments (qt = M^T q into the workspace, M at the
    // segment ends), up to the horizon, then over the rest where M is not yet zero.
    RunParams pb = pa;
    pb.init = nullptr;
    pb.init_idx = nullptr;
    pb.zero_v = true;
    pb.identity_init = true;
    pb.o = qt;
    pb.fin = mtr;
    pb.max_chunks = kHorizon / 64;
    pb.skip = skip;
    pb.out_gate = nullptr;  // its "o" is qt
    if ((e = launch_tc_prefill(pb, s)) != cudaSuccess) return e;
    seg_done_kernel<<<(unsigned)(S * H), 256, 0, s>>>(mtr, skip, done);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pb.max_chunks = 0;
    pb.skip = done;
    if ((e = launch_tc_prefill(pb, s)) != cudaSuccess) return e;
    // Start states of the later segments and the final states.
    seg_scan_kernel<<<(unsigned)(n * H), 256, kScanSmem, s>>>(mtr, sloc, nullptr, p.fin, nullptr, p.fin_idx, p.pool,
                                                              p.err, sst, 0, H, seg_first);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // o += S_start^T qt on the later segments.
    CUtensorMap qt_map;
    if (!encode_row_tile_map(&qt_map, qt, (long long)T, H)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)kTilesPerCta, (unsigned)S, (unsigned)H);
    seg_correct_kernel<<<grid, 128, kCorrectSmem, s>>>(qt_map, sst, done, static_cast<__nv_bfloat16 *>(p.o),
                                                       static_cast<const __nv_bfloat16 *>(p.out_gate), T, H, 0, 1, 0,
                                                       seg_cu, is_first, p.err);
    return cudaGetLastError();
}

cudaError_t launch_segmented_prefill(const RunParams &p, int B, void *workspace, size_t workspace_bytes,
                                     cudaStream_t s) {
    const int T = p.T, H = p.H;
    const Plan pl = make_plan(B, T, H);
    if (pl.P < 2 || workspace_bytes < pl.bytes || !workspace) return cudaErrorInvalidValue;
    cudaError_t e = set_segmented_attributes();
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *cu = reinterpret_cast<int32_t *>(ws + pl.off_cu);
    __nv_bfloat16 *qt = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_qt);
    float *sloc = reinterpret_cast<float *>(ws + pl.off_sloc);
    float *mtr = reinterpret_cast<float *>(ws + pl.off_mtr);
    __nv_bfloat16 *sst = reinterpret_cast<__nv_bfloat16 *>(ws + pl.off_sst);
    uint8_t *done = ws + pl.off_done;
    const int segs = B * pl.P;

    seg_bounds_kernel<<<1, 256, 0, s>>>(cu, B, T, pl.P, pl.Ls);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // Pass 1: the segments from a zero state (o^loc into o, S^loc into the workspace).
    RunParams pa = p;
    pa.cu_seqlens = cu;
    pa.n_seqs = segs;
    pa.T = B * T;
    pa.init = nullptr;
    pa.fin = sloc;
    pa.zero_v = false;
    pa.identity_init = false;
    pa.max_chunks = 0;
    pa.skip = nullptr;
    pa.init_idx = nullptr;
    pa.fin_idx = nullptr;
    if ((e = launch_tc_prefill(pa, s)) != cudaSuccess) return e;
    // Pass 2: v = 0 from the identity (qt = M^T q into the workspace, M at the segment ends): first
    // up to the horizon, then, for the pairs whose M is not zero there, over the whole segment.
    RunParams pb = pa;
    pb.zero_v = true;
    pb.identity_init = true;
    pb.o = qt;
    pb.fin = mtr;
    pb.max_chunks = kHorizon / 64;
    pb.out_gate = nullptr;  // its "o" is qt
    pb.qk_l2norm = p.qk_l2norm;
    if ((e = launch_tc_prefill(pb, s)) != cudaSuccess) return e;
    seg_done_kernel<<<(unsigned)(segs * H), 256, 0, s>>>(mtr, nullptr, done);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pb.max_chunks = 0;
    pb.skip = done;
    if ((e = launch_tc_prefill(pb, s)) != cudaSuccess) return e;
    // Start states of the segments and the final state.
    seg_scan_kernel<<<(unsigned)(B * H), 256, kScanSmem, s>>>(mtr, sloc, p.init, p.fin, p.init_idx, p.fin_idx,
                                                              p.pool, p.err, sst, pl.P, H, nullptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // o += S_start^T qt, skipped for segment 0 when the initial state is zero.
    CUtensorMap qt_map;
    if (!encode_row_tile_map(&qt_map, qt, (long long)B * T, H)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((pl.Ls + CT * kTilesPerCta - 1) / (CT * kTilesPerCta)), (unsigned)segs, (unsigned)H);
    seg_correct_kernel<<<grid, 128, kCorrectSmem, s>>>(qt_map, sst, done, static_cast<__nv_bfloat16 *>(p.o),
                                                       static_cast<const __nv_bfloat16 *>(p.out_gate), T, H,
                                                       pl.Ls, pl.P, p.init ? 0 : 1, nullptr, nullptr, p.err);
    return cudaGetLastError();
}

}  // namespace kda
