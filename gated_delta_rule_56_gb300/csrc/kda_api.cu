// kda_api.cu -- the C ABI of libkda.so: host-side validation and kernel dispatch.
//
// Entry points and their contracts are declared in include/kda.h. Every check that can be
// made on the host is made here before anything is queued; the kernels only see arguments
// that passed. Conditions only the device can see are OR-ed into a per-device error word.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kda_internal.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

__device__ unsigned g_error_word;  // one per device: bits kErrBadSeqlens | kErrTimeout

thread_local char g_last_error[512];

kda_status fail(kda_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

kda_status ok() {
    g_last_error[0] = '\0';
    return KDA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head(int dk, int dv) { return dk == dv && (dk == 32 || dk == 64 || dk == 128); }

kda_status check_head(int dk, int dv) {
    if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARG, "dk=%d dv=%d must be positive", dk, dv);
    if (!supported_head(dk, dv))
        return fail(KDA_ERR_UNSUPPORTED, "head sizes dk=%d dv=%d: supported dk == dv in {32, 64, 128}",
                    dk, dv);
    return KDA_OK;
}

kda_status check_dtype(kda_dtype dt) {
    if (dt != KDA_BF16 && dt != KDA_F32) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    return KDA_OK;
}

kda_status check_ptr(const void *p, const char *name, bool need_align) {
    if (!p) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", name);
    if (need_align && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return KDA_OK;
}

// One thread waits, bounded, on an mbarrier phase that nothing completes (count 1, no arrival),
// with the library's own bounded wait, and records the time-out like a pipeline wait would.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        if (!tc::mbar_wait(&bar, 0, limit_ns)) atomicOr(&g_error_word, kErrTimeout);
    }
}

kda_status launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

// Scratch of kda_prefill_noalloc: one array per device, placed when the module loads, so that
// the call allocates nothing. 32 MiB holds the split of about 100 K token-heads.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

struct StaticScratch {
    void *addr = nullptr;
    cudaEvent_t last = nullptr;  // recorded after the latest call that used the scratch
};

// Looks up the scratch address and creates the ordering event once per device.
StaticScratch *static_scratch(int dev) {
    static StaticScratch slots[256];
    if (dev < 0 || dev >= 256) return nullptr;
    StaticScratch &sc = slots[dev];
    if (!sc.addr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&sc.last, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        sc.addr = addr;
    }
    return &sc;
}

std::mutex g_static_scratch_mu;

// Longest-first order of packed sequences: one CTA sorts (length, index) keys (length
// descending, index ascending among equals) with a bitonic network in shared memory. The
// tensor-core kernel then starts the longest sequences' CTAs first, so the last CTAs to start are
// short ones and the tail of the launch is short. A malformed cu_seqlens still gives a
// permutation (its lengths are clamped); the kernel reports it as before.
constexpr int kSortThreads = 1024;
__global__ void __launch_bounds__(kSortThreads) order_by_length_kernel(const int32_t *__restrict__ cu, int n,
                                                                        int32_t *__restrict__ order) {
    __shared__ unsigned long long key[kMaxOrderedSeqs];
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = threadIdx.x; i < m; i += kSortThreads) {
        if (i < n) {
            const long long len = (long long)cu[i + 1] - cu[i];
            const unsigned inv = 0x7fffffffu - (unsigned)(len < 0 ? 0 : (len > 0x7fffffff ? 0x7fffffff : len));
            key[i] = ((unsigned long long)inv << 32) | (unsigned)i;
        } else {
            key[i] = ~0ull;
        }
    }
    __syncthreads();
    for (int size = 2; size <= m; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < m; i += kSortThreads) {
                const int jx = i ^ stride;
                if (jx > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long a = key[i], b = key[jx];
                    if ((a > b) == up) {
                        key[i] = b;
                        key[jx] = a;
                    }
                }
            }
            __syncthreads();
        }
    for (int i = threadIdx.x; i < n; i += kSortThreads) order[i] = (int32_t)(key[i] & 0xffffffffu);
}

}  // namespace

size_t order_workspace_bytes(kda_dtype dtype, int dk, int dv, int n_seqs) {
    if (dtype != KDA_BF16 || dk != dv || (dk != 32 && dk != 64 && dk != 128) || n_seqs < 2 ||
        n_seqs > kMaxOrderedSeqs)
        return 0;
    return ((size_t)n_seqs * sizeof(int32_t) + 255) / 256 * 256;
}

cudaError_t launch_order_by_length(const int32_t *cu_seqlens, int n_seqs, int32_t *order, cudaStream_t s) {
    order_by_length_kernel<<<1, kSortThreads, 0, s>>>(cu_seqlens, n_seqs, order);
    return cudaGetLastError();
}

unsigned *device_error_word() {
    static std::mutex mu;
    static unsigned *words[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!words[dev]) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return nullptr;
        words[dev] = static_cast<unsigned *>(addr);
    }
    return words[dev];
}

}  // namespace kda

using namespace kda;

namespace kda {
namespace {

// The caller's options, read up to the size it was compiled with (later fields keep their
// defaults), and checked. NULL means all defaults.
kda_status read_options(const kda_options *user, kda_options &opt) {
    opt = kda_options{};
    opt.struct_size = sizeof(kda_options);
    if (!user) return KDA_OK;
    if (user->struct_size < sizeof(size_t) || user->struct_size > 4096)
        return fail(KDA_ERR_INVALID_ARG, "kda_options.struct_size=%zu is not the size of a kda_options",
                    user->struct_size);
    const size_t n = user->struct_size < sizeof(kda_options) ? user->struct_size : sizeof(kda_options);
    memcpy(&opt, user, n);
    opt.struct_size = sizeof(kda_options);
    if (!(opt.gate_bound == 0.f || (opt.gate_bound > 0.f && opt.gate_bound <= 1e4f)))
        return fail(KDA_ERR_INVALID_ARG, "gate_bound=%g must be 0 or in (0, 1e4]", (double)opt.gate_bound);
    if (opt.initial_state_indices || opt.final_state_indices) {
        if (opt.state_pool_size <= 0)
            return fail(KDA_ERR_INVALID_ARG, "state_pool_size=%d must be positive when state indices are given",
                        opt.state_pool_size);
        if ((reinterpret_cast<uintptr_t>(opt.initial_state_indices) & 3u) ||
            (reinterpret_cast<uintptr_t>(opt.final_state_indices) & 3u))
            return fail(KDA_ERR_INVALID_ARG, "state index arrays must be 4-byte aligned");
    }
    if (opt.out_gate && !aligned16(opt.out_gate))
        return fail(KDA_ERR_INVALID_ARG, "out_gate is not 16-byte aligned");
    return KDA_OK;
}

kda_options gate_only(float gate_bound) {
    kda_options opt{};
    opt.struct_size = sizeof(kda_options);
    opt.gate_bound = gate_bound;
    return opt;
}

// Workspace a prefill call can use on a GPU with `sms` SMs: packed sequences (cu_seqlens given)
// are split along the sequence when fewer of them than SMs / H are long enough, else they take the
// longest-first launch order; unpacked ones the split along the sequence.
size_t prefill_workspace_bytes_for(kda_dtype dtype, int B, int T, int H, int dk, int dv, bool packed, int n_seqs,
                                   int sms) {
    if (B < 0 || T < 0 || H < 0 || sms < 0) return 0;
    if (packed) {
        if (B != 1) return 0;
        const size_t split = segmented_packed_workspace_bytes_for(dtype, n_seqs, T, H, dk, dv, sms);
        return split ? split : order_workspace_bytes(dtype, dk, dv, n_seqs);
    }
    if (dtype != KDA_BF16 || dk != 128 || dv != 128) return 0;
    int P = 0, Ls = 0;
    size_t bytes = 0;
    segmented_plan_for(B, T, H, sms, &P, &Ls, &bytes);
    return bytes;
}

// SMs of the current device (0 when none is visible).
int current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        sms = 0;
    }
    return sms;
}

// The same on the current device.
size_t prefill_workspace_bytes(kda_dtype dtype, int B, int T, int H, int dk, int dv, bool packed, int n_seqs) {
    return prefill_workspace_bytes_for(dtype, B, T, H, dk, dv, packed, n_seqs, current_sms());
}

// The common body of kda_prefill, kda_prefill_gated and kda_prefill_ex.
kda_status prefill_impl(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q,
                        const void *k, const void *v, const void *g, const void *beta,
                        const int32_t *cu_seqlens, int n_seqs, const float *initial_state, void *o,
                        float *final_state, const kda_options &opt, void *workspace, size_t workspace_bytes,
                        kda_stream_t stream) {
    kda_status st;
    if ((st = check_dtype(dtype)) != KDA_OK) return st;
    if (B < 0 || T < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "negative size B=%d T=%d H=%d", B, T, H);
    if ((st = check_head(dk, dv)) != KDA_OK) return st;
    if (cu_seqlens) {
        if (B != 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens requires B == 1 (got B=%d)", B);
        if (n_seqs < 0) return fail(KDA_ERR_INVALID_ARG, "n_seqs=%d is negative", n_seqs);
        if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
    } else {
        n_seqs = B;
    }
    const long long rows = (long long)B * T;
    if ((long long)n_seqs * H > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "too many (sequence, head) pairs");
    if (rows * H * (long long)(dk > dv ? dk : dv) > (1LL << 46))
        return fail(KDA_ERR_INVALID_ARG, "tensor too large");
    if (rows > 0) {
        if ((st = check_ptr(q, "q", true)) || (st = check_ptr(k, "k", true)) ||
            (st = check_ptr(v, "v", true)) || (st = check_ptr(g, "g", true)) ||
            (st = check_ptr(o, "o", true)) || (st = check_ptr(beta, "beta", false)))
            return st;
        if ((reinterpret_cast<uintptr_t>(beta) & (dtype == KDA_BF16 ? 1u : 3u)) != 0)
            return fail(KDA_ERR_INVALID_ARG, "beta is not aligned to its element size");
    }
    if (initial_state && !aligned16(initial_state))
        return fail(KDA_ERR_INVALID_ARG, "initial_state is not 16-byte aligned");
    if (final_state && !aligned16(final_state))
        return fail(KDA_ERR_INVALID_ARG, "final_state is not 16-byte aligned");
    if ((long long)n_seqs * H == 0) return ok();

    RunParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.cu_seqlens = cu_seqlens;
    p.init = initial_state;
    p.fin = final_state;
    p.o = o;
    p.T = T;
    p.H = H;
    p.dk = dk;
    p.n_seqs = n_seqs;
    p.err = device_error_word();
    p.gate_bound = opt.gate_bound;
    p.qk_l2norm = opt.qk_l2norm != 0;
    if (opt.initial_state_indices && !initial_state)
        return fail(KDA_ERR_INVALID_ARG, "initial_state_indices given without initial_state (the pool)");
    if (opt.final_state_indices && !final_state)
        return fail(KDA_ERR_INVALID_ARG, "final_state_indices given without final_state (the pool)");
    p.init_idx = opt.initial_state_indices;
    p.fin_idx = opt.final_state_indices;
    p.pool = opt.state_pool_size;
    p.out_gate = opt.out_gate;
    if (!p.err) return fail(KDA_ERR_CUDA, "cannot reach the device error word: %s",
                            cudaGetErrorString(cudaGetLastError()));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_prefill_supported(dtype, dk, dv, p)) {
        // Few packed sequences: split the long ones along the sequence when the caller gave the workspace.
        const size_t pk_bytes =
            cu_seqlens ? segmented_packed_workspace_bytes_for(dtype, n_seqs, T, H, dk, dv, current_sms()) : 0;
        if (pk_bytes && workspace && workspace_bytes >= pk_bytes && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)
            return launched(launch_segmented_packed_prefill(p, workspace, workspace_bytes, s), "segmented packed prefill");
        // Packed sequences: start the longest first when the caller gave the workspace for the order.
        const size_t ord_bytes = cu_seqlens ? order_workspace_bytes(dtype, dk, dv, n_seqs) : 0;
        if (ord_bytes && workspace && workspace_bytes >= ord_bytes &&
            (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0) {
            int32_t *order = static_cast<int32_t *>(workspace);
            const cudaError_t e = launch_order_by_length(cu_seqlens, n_seqs, order, s);
            if (e != cudaSuccess) return launched(e, "sequence order");
            p.order = order;
        }
        // A few long sequences: split them along the sequence when the caller gave the workspace.
        const size_t seg_bytes = segmented_workspace_bytes(dtype, B, T, H, dk, dv, cu_seqlens != nullptr);
        if (seg_bytes && workspace && workspace_bytes >= seg_bytes &&
            (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)
            return launched(launch_segmented_prefill(p, B, workspace, workspace_bytes, s), "segmented prefill");
        return launched(launch_tc_prefill(p, s), "tensor-core prefill");
    }
    if (tf32_prefill_supported(dtype, dk, dv, p)) return launched(launch_tf32_prefill(p, s), "tf32 tensor-core prefill");
    return launched(launch_recurrent(dtype, dk, dv, p, s), "recurrent prefill");
}

// The common body of kda_decode_step, kda_decode_step_gated and kda_decode_step_ex.
kda_status decode_impl(kda_dtype dtype, int N, int H, int dk, int dv, const void *q, const void *k,
                       const void *v, const void *g, const void *beta, float *state, void *o,
                       const kda_options &opt, kda_stream_t stream) {
    kda_status st;
    if ((st = check_dtype(dtype)) != KDA_OK) return st;
    if (N < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "negative size N=%d H=%d", N, H);
    if ((st = check_head(dk, dv)) != KDA_OK) return st;
    if ((long long)N * H == 0) return ok();
    if ((long long)N * H > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "too many (sequence, head) pairs");
    if ((st = check_ptr(q, "q", true)) || (st = check_ptr(k, "k", true)) || (st = check_ptr(v, "v", true)) ||
        (st = check_ptr(g, "g", true)) || (st = check_ptr(o, "o", true)) ||
        (st = check_ptr(state, "state", true)) || (st = check_ptr(beta, "beta", false)))
        return st;
    if ((reinterpret_cast<uintptr_t>(beta) & (dtype == KDA_BF16 ? 1u : 3u)) != 0)
        return fail(KDA_ERR_INVALID_ARG, "beta is not aligned to its element size");

    RunParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.cu_seqlens = nullptr;
    p.init = state;
    p.fin = state;
    p.o = o;
    p.T = 1;
    p.H = H;
    p.dk = dk;
    p.n_seqs = N;
    p.err = device_error_word();
    p.gate_bound = opt.gate_bound;
    p.qk_l2norm = opt.qk_l2norm != 0;
    if (opt.final_state_indices && !opt.initial_state_indices)
        return fail(KDA_ERR_INVALID_ARG, "decode: final_state_indices needs initial_state_indices");
    p.init_idx = opt.initial_state_indices;
    p.fin_idx = opt.final_state_indices ? opt.final_state_indices : opt.initial_state_indices;
    p.pool = opt.state_pool_size;
    p.out_gate = opt.out_gate;
    if (!p.err) return fail(KDA_ERR_CUDA, "cannot reach the device error word");
    return launched(launch_recurrent(dtype, dk, dv, p, reinterpret_cast<cudaStream_t>(stream)), "decode step");
}

}  // namespace
}  // namespace kda

extern "C" {

int kda_version(void) { return 2 * 10000 + 0 * 100 + 0; }

kda_status kda_selftest_wait_timeout(uint64_t limit_ns, kda_stream_t stream) {
    if (limit_ns < 1 || limit_ns > 1000000000ull)
        return fail(KDA_ERR_INVALID_ARG, "limit_ns=%llu must be in [1, 1e9]", (unsigned long long)limit_ns);
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
    return launched(cudaGetLastError(), "wait_timeout_kernel");
}

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

const char *kda_last_error(void) { return g_last_error; }

size_t kda_prefill_workspace_size(kda_dtype dtype, int B, int T, int H, int dk, int dv, const int32_t *cu_seqlens,
                                  int n_seqs) {
    return prefill_workspace_bytes(dtype, B, T, H, dk, dv, cu_seqlens != nullptr, n_seqs);
}

size_t kda_prefill_workspace_size_for(kda_dtype dtype, int B, int T, int H, int dk, int dv, const int32_t *cu_seqlens,
                                      int n_seqs, int sm_count) {
    return prefill_workspace_bytes_for(dtype, B, T, H, dk, dv, cu_seqlens != nullptr, n_seqs, sm_count);
}

kda_status kda_prefill_split_plan(int B, int T, int H, int sm_count, int *segments, int *segment_rows,
                                  size_t *workspace_bytes) {
    if (!segments || !segment_rows || !workspace_bytes)
        return fail(KDA_ERR_INVALID_ARG, "NULL output pointer");
    if (B < 0 || T < 0 || H < 0 || sm_count < 0)
        return fail(KDA_ERR_INVALID_ARG, "negative size B=%d T=%d H=%d sm_count=%d", B, T, H, sm_count);
    segmented_plan_for(B, T, H, sm_count, segments, segment_rows, workspace_bytes);
    return ok();
}

kda_status kda_prefill(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q,
                       const void *k, const void *v, const void *g, const void *beta,
                       const int32_t *cu_seqlens, int n_seqs, const float *initial_state, void *o,
                       float *final_state, void *workspace, size_t workspace_bytes,
                       kda_stream_t stream) {
    return prefill_impl(dtype, B, T, H, dk, dv, q, k, v, g, beta, cu_seqlens, n_seqs, initial_state, o,
                        final_state, gate_only(0.f), workspace, workspace_bytes, stream);
}

kda_status kda_prefill_ex(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q, const void *k,
                          const void *v, const void *g, const void *beta, const int32_t *cu_seqlens, int n_seqs,
                          const float *initial_state, void *o, float *final_state, const kda_options *options,
                          void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    kda_options opt;
    const kda_status st = read_options(options, opt);
    if (st != KDA_OK) return st;
    return prefill_impl(dtype, B, T, H, dk, dv, q, k, v, g, beta, cu_seqlens, n_seqs, initial_state, o,
                        final_state, opt, workspace, workspace_bytes, stream);
}

kda_status kda_prefill_gated(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q,
                             const void *k, const void *v, const void *gate_logits, const void *beta,
                             const int32_t *cu_seqlens, int n_seqs, const float *initial_state, void *o,
                             float *final_state, float gate_bound, void *workspace, size_t workspace_bytes,
                             kda_stream_t stream) {
    if (!(gate_bound > 0.f && gate_bound <= 1e4f))
        return fail(KDA_ERR_INVALID_ARG, "gate_bound=%g must be in (0, 1e4]", (double)gate_bound);
    return prefill_impl(dtype, B, T, H, dk, dv, q, k, v, gate_logits, beta, cu_seqlens, n_seqs, initial_state,
                        o, final_state, gate_only(gate_bound), workspace, workspace_bytes, stream);
}

kda_status kda_prefill_debug_dump(int B, int T, int H, const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const float *initial_state, void *o, float *final_state,
                                  float *dump, int dump_chunks, kda_stream_t stream) {
    if (B < 1 || T < 1 || H < 1 || dump_chunks < 0)
        return fail(KDA_ERR_INVALID_ARG, "B=%d T=%d H=%d dump_chunks=%d", B, T, H, dump_chunks);
    if ((long long)B * T > 0x7fffffffLL - 64 || (long long)B * H > 0x7fffffffLL)
        return fail(KDA_ERR_INVALID_ARG, "too large");
    kda_status st;
    if ((st = check_ptr(q, "q", true)) || (st = check_ptr(k, "k", true)) || (st = check_ptr(v, "v", true)) ||
        (st = check_ptr(g, "g", true)) || (st = check_ptr(o, "o", true)) || (st = check_ptr(beta, "beta", false)) ||
        (st = check_ptr(dump, "dump", true)))
        return st;
    if ((reinterpret_cast<uintptr_t>(beta) & 1u) || (initial_state && !aligned16(initial_state)) ||
        (final_state && !aligned16(final_state)))
        return fail(KDA_ERR_INVALID_ARG, "misaligned beta or state");
    RunParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.init = initial_state;
    p.fin = final_state;
    p.o = o;
    p.T = T;
    p.H = H;
    p.dk = 128;
    p.n_seqs = B;
    p.err = device_error_word();
    p.dump = dump;
    p.dump_chunks = dump_chunks;
    if (!p.err) return fail(KDA_ERR_CUDA, "cannot reach the device error word");
    if (!tc_prefill_supported(KDA_BF16, 128, 128, p))
        return fail(KDA_ERR_UNSUPPORTED, "the tensor-core prefill is not available");
    return launched(launch_tc_prefill(p, reinterpret_cast<cudaStream_t>(stream)), "tensor-core prefill (dump)");
}

size_t kda_prefill_noalloc_capacity(void) { return kStaticScratchBytes; }

kda_status kda_prefill_noalloc(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q,
                               const void *k, const void *v, const void *g, const void *beta,
                               const int32_t *cu_seqlens, int n_seqs, const float *initial_state, void *o,
                               float *final_state, kda_stream_t stream) {
    const size_t need = prefill_workspace_bytes(dtype, B, T, H, dk, dv, cu_seqlens != nullptr, n_seqs);
    if (need > kStaticScratchBytes)
        return fail(KDA_ERR_UNSUPPORTED, "this call needs %zu bytes of scratch; the static scratch holds %zu",
                    need, kStaticScratchBytes);
    if (need == 0)
        return prefill_impl(dtype, B, T, H, dk, dv, q, k, v, g, beta, cu_seqlens, n_seqs, initial_state, o,
                            final_state, gate_only(0.f), nullptr, 0, stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    StaticScratch *sc = static_scratch(dev);
    if (!sc) return fail(KDA_ERR_CUDA, "static scratch: %s", cudaGetErrorString(cudaGetLastError()));
    // Calls on different streams share the scratch: each waits for the previous one's work.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((e = cudaStreamWaitEvent(s, sc->last, 0)) != cudaSuccess)
        return fail(KDA_ERR_CUDA, "ordering on the static scratch: %s", cudaGetErrorString(e));
    const kda_status st = prefill_impl(dtype, B, T, H, dk, dv, q, k, v, g, beta, cu_seqlens, n_seqs,
                                       initial_state, o, final_state, gate_only(0.f), sc->addr, kStaticScratchBytes,
                                       stream);
    // Recorded whatever the status: a call that failed part-way may have queued kernels that use
    // the scratch, and the next call must still wait for them. Its own failure is reported first.
    e = cudaEventRecord(sc->last, s);
    if (st != KDA_OK) return st;
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "ordering on the static scratch: %s", cudaGetErrorString(e));
    return st;
}

size_t kda_backward_workspace_size(kda_dtype dtype, int B, int T, int H, int dk, int dv, int n_seqs) {
    (void)dtype;
    if (B < 0 || T < 0 || H <= 0 || dk != dv || dk <= 0) return 0;
    return backward_workspace_bytes((int)((long long)B * T > 0x7fffffffLL ? 0x7fffffff : (long long)B * T),
                                    n_seqs > B ? n_seqs : B, H, dk);
}

kda_status kda_backward(kda_dtype dtype, int B, int T, int H, int dk, int dv, const void *q, const void *k,
                        const void *v, const void *g, const void *beta, const int32_t *cu_seqlens, int n_seqs,
                        const float *initial_state, const void *d_o, const float *d_final_state, float *dq,
                        float *dk_out, float *dv_out, float *dg, float *dbeta, float *d_initial_state,
                        void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    kda_status st;
    if ((st = check_dtype(dtype)) != KDA_OK) return st;
    if (B < 0 || T < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "negative size B=%d T=%d H=%d", B, T, H);
    if ((st = check_head(dk, dv)) != KDA_OK) return st;
    if (cu_seqlens) {
        if (B != 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens requires B == 1 (got B=%d)", B);
        if (n_seqs < 0) return fail(KDA_ERR_INVALID_ARG, "n_seqs=%d is negative", n_seqs);
        if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
    } else {
        n_seqs = B;
    }
    const long long rows = (long long)B * T;
    if ((long long)n_seqs * H > 0x7fffffffLL || rows > 0x7fffffffLL)
        return fail(KDA_ERR_INVALID_ARG, "too many rows or (sequence, head) pairs");
    if ((long long)n_seqs * H == 0) return ok();
    if (rows > 0) {
        if ((st = check_ptr(q, "q", true)) || (st = check_ptr(k, "k", true)) || (st = check_ptr(v, "v", true)) ||
            (st = check_ptr(g, "g", true)) || (st = check_ptr(beta, "beta", false)) ||
            (st = check_ptr(d_o, "d_o", true)) || (st = check_ptr(dq, "dq", true)) ||
            (st = check_ptr(dk_out, "dk", true)) || (st = check_ptr(dv_out, "dv", true)) ||
            (st = check_ptr(dg, "dg", true)) || (st = check_ptr(dbeta, "dbeta", false)))
            return st;
        if ((reinterpret_cast<uintptr_t>(beta) & (dtype == KDA_BF16 ? 1u : 3u)) != 0)
            return fail(KDA_ERR_INVALID_ARG, "beta is not aligned to its element size");
        if ((reinterpret_cast<uintptr_t>(dbeta) & 3u) != 0) return fail(KDA_ERR_INVALID_ARG, "dbeta is not 4-byte aligned");
    }
    if ((initial_state && !aligned16(initial_state)) || (d_final_state && !aligned16(d_final_state)) ||
        (d_initial_state && !aligned16(d_initial_state)))
        return fail(KDA_ERR_INVALID_ARG, "state pointers must be 16-byte aligned");
    const size_t need = backward_workspace_bytes((int)rows, n_seqs, H, dk);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(KDA_ERR_INVALID_ARG, "workspace: %zu bytes at a 16-byte aligned address needed, got %zu",
                    need, workspace ? workspace_bytes : (size_t)0);
    RunParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.cu_seqlens = cu_seqlens;
    p.init = initial_state;
    p.T = T;
    p.H = H;
    p.dk = dk;
    p.n_seqs = n_seqs;
    p.err = device_error_word();
    if (!p.err) return fail(KDA_ERR_CUDA, "cannot reach the device error word");
    return launched(launch_backward(dtype, dk, p, d_o, d_final_state, dq, dk_out, dv_out, dg, dbeta,
                                    d_initial_state, workspace, reinterpret_cast<cudaStream_t>(stream)),
                    "backward");
}

kda_status kda_decode_step(kda_dtype dtype, int N, int H, int dk, int dv, const void *q, const void *k,
                           const void *v, const void *g, const void *beta, float *state, void *o,
                           kda_stream_t stream) {
    return decode_impl(dtype, N, H, dk, dv, q, k, v, g, beta, state, o, gate_only(0.f), stream);
}

kda_status kda_decode_step_ex(kda_dtype dtype, int N, int H, int dk, int dv, const void *q, const void *k,
                              const void *v, const void *g, const void *beta, float *state, void *o,
                              const kda_options *options, kda_stream_t stream) {
    kda_options opt;
    const kda_status st = read_options(options, opt);
    if (st != KDA_OK) return st;
    return decode_impl(dtype, N, H, dk, dv, q, k, v, g, beta, state, o, opt, stream);
}

kda_status kda_decode_step_gated(kda_dtype dtype, int N, int H, int dk, int dv, const void *q, const void *k,
                                 const void *v, const void *gate_logits, const void *beta, float *state, void *o,
                                 float gate_bound, kda_stream_t stream) {
    if (!(gate_bound > 0.f && gate_bound <= 1e4f))
        return fail(KDA_ERR_INVALID_ARG, "gate_bound=%g must be in (0, 1e4]", (double)gate_bound);
    return decode_impl(dtype, N, H, dk, dv, q, k, v, gate_logits, beta, state, o, gate_only(gate_bound), stream);
}

kda_status kda_check_status(kda_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
    if (e == cudaSuccess && word) e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "error word: %s", cudaGetErrorString(e));
    if (word & kErrTimeout) return fail(KDA_ERR_TIMEOUT, "a device-side wait gave up (error word 0x%x)", word);
    if (word & kErrBadIndex)
        return fail(KDA_ERR_INVALID_ARG, "a state index is at or past the pool end (error word 0x%x)", word);
    if (word & kErrBadSeqlens)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not a non-decreasing list ending at T (error word 0x%x)", word);
    return ok();
}

}  // extern "C"
