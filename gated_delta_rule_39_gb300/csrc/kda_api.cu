// Host side of the C ABI declared in include/kda.h: argument validation,
// stream-ordered scratch memory, kernel launches, error word, launch timing.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

// cudaError_t behind the calling thread's most recent KDA_ERR_LAUNCH / ALLOC / CUDA
thread_local int t_last_cuda_error = 0;
// record a CUDA failure, clear the runtime's (non-sticky) last error, pass `status` on
int cuda_fail(int status, cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    return status;
}

// Device-side error word (one per device: every device that loads the module
// holds its own instance).  Kernels receive its address.
__device__ int g_error_word;

constexpr int kMaxDevices = 64;
// A 16-token chunk of gates at the bound spans 16 * 5.4 / ln 2 = 124.6 bits of decay.
// The in-chunk factors 2^G of its last rows then stay normal fp32 numbers; much
// closer to 2^-126 the products q 2^G, k 2^G fall into the subnormal range and lose
// precision, and at -5.5 (126.96 bits) 2^G itself underflows.
constexpr float kLowerBoundMin = -5.4f;

struct DeviceInfo {
    bool ready = false;
    bool arch_ok = false;
    int sms = 0;   // streaming multiprocessors
    int* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_setup(int* dev_out, int** err_out, int* sms_out = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(KDA_ERR_CUDA, cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
        d.arch_ok = (major == 10 && minor == 3);
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
        d.err = static_cast<int*>(p);
        // keep freed scratch in the device's default pool instead of returning
        // it to the driver at every synchronisation
        cudaMemPool_t pool;
        if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
            uint64_t thr = UINT64_MAX;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
        }
        d.ready = true;
    }
    *dev_out = dev;
    *err_out = d.err;
    if (sms_out) *sms_out = d.sms;
    return d.arch_ok ? KDA_OK : KDA_ERR_ARCH;
}

// ---- launch timing ------------------------------------------------------------
struct TimingRecord {
    int kernel;
    cudaEvent_t start, stop;
};
struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<TimingRecord> pending;
    std::vector<cudaEvent_t> free_events;
    double total_ms[KDA_NUM_KERNELS] = {};
    long long launches[KDA_NUM_KERNELS] = {};
} g_prof;

cudaEvent_t prof_event() {
    if (!g_prof.free_events.empty()) {
        cudaEvent_t e = g_prof.free_events.back();
        g_prof.free_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

template <class F>
cudaError_t timed_launch(int kernel, cudaStream_t s, F&& launch) {
    bool on;
    {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        on = g_prof.on;
    }
    if (!on) return launch();
    cudaEvent_t a, b;
    {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        a = prof_event();
        b = prof_event();
    }
    cudaEventRecord(a, s);
    cudaError_t e = launch();
    cudaEventRecord(b, s);
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.pending.push_back({kernel, a, b});
    return e;
}

// ---- scratch ------------------------------------------------------------------
constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Scratch of one call: the varlen sequence map (longest-first order, valid flag and
// the unit counter of a persistent launch); fixed-length calls need none unless they
// are split into segments.
size_t scratch_bytes(int N, bool varlen) {
    return varlen ? align_up(sizeof(int) * ((size_t)N + 2)) : 0;
}

// Varlen calls whose sequences average at most this many tokens run persistent CTAs
// (one per SM, units taken longest first from a device counter, pipelines carried from
// unit to unit) when they have more (sequence, head) units than SMs.  Measured on
// GB300 against one CTA per unit: 1.9x at 8-16 tokens, 1.7x at 32, 1.5x at 64, 1.3x
// at 128 and 1.2x at 200 tokens per sequence, but 3-9 % slower at 700-1,000 tokens,
// where a CTA's start-up is a small part of its unit.
constexpr int kPersistMaxAvgTokens = 256;

// ---- sequence split (kda_split.cu) -----------------------------------------------
// Shortest segment the automatic split makes: 64 chunks, so that the two launches,
// the combine step and each CTA's pipeline fill stay small against a segment's time.
constexpr int kSplitMinTokens = 1024;

// Segments for a fixed-length call: `requested` 0 picks them (the largest s whose
// window-0 units, (2s - 3) B H, fit on the device's SMs in one wave, with at least
// kSplitMinTokens per segment; 1 when that gives fewer than 3), 1 is one pass, s >= 2
// is s segments of whole chunks, at most one per chunk.  Returns 0 if `requested`
// cannot be met.
int plan_segments(int B, int T, int H, int requested, int sms) {
    if (requested == 1) return 1;
    if (requested >= 2) return requested <= (T + kChunk - 1) / kChunk ? requested : 0;
    const double units = (double)B * H;
    if (sms <= 0 || T < 1 || units <= 0) return 1;
    int s = (int)(((double)sms / units + 3.0) / 2.0);
    s = std::min(s, T / kSplitMinTokens);
    return s >= 3 ? s : 1;
}

// Scratch of a split call (fp32 states of every unit; see kda_split.cu): window 0's
// initial states (reused for window 1's end states), window 0's end states, window 1's
// initial states, and 16 zero rows of values.
struct SplitScratch {
    size_t init0, end0, init1, zero, total;
};
SplitScratch split_layout(int N, int H, int s) {
    SplitScratch L{};
    if (s < 2) return L;
    const size_t st = (size_t)kDim * kDim * sizeof(float) * N * H;
    L.init0 = 0;
    L.end0 = align_up(st * (2 * s - 3));
    L.init1 = L.end0 + align_up(st * (2 * s - 3));
    L.zero = L.init1 + align_up(st * (s - 1));
    L.total = L.zero + align_up((size_t)kChunk * H * kDim * 2);
    return L;
}
size_t split_bytes(int N, int H, int s) { return split_layout(N, H, s).total; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Host-side checks shared by kda_fwd and kda_fwd_host; no CUDA call.
int validate(const void* q, const void* k, const void* v, const void* g, const void* beta,
             float scale, const void* out, const float* A_log, const float* dt_bias,
             float lower_bound, const void* s0, int s0_dtype, const void* s1, int s1_dtype,
             const int32_t* cu, int num_seqs, int B, int T, int H, int K, int V, bool check_align) {
    if (K != kDim || V != kDim) return KDA_ERR_UNSUPPORTED_DIM;
    if (B < 1 || T < 0 || H < 1) return KDA_ERR_SHAPE;
    if (cu) {
        if (B != 1 || num_seqs < 1) return KDA_ERR_SHAPE;
    }
    const long long tok = (long long)B * T;
    if (tok * H * kDim >= (1LL << 31)) return KDA_ERR_SHAPE;
    if (cu && (long long)num_seqs * H * kDim * kDim >= (1LL << 40)) return KDA_ERR_SHAPE;
    if (tok > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (!A_log || !dt_bias) return KDA_ERR_NULL;
    if (s0 && s0_dtype != KDA_BF16 && s0_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (s1 && s1_dtype != KDA_BF16 && s1_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!std::isfinite(scale)) return KDA_ERR_ARG;
    if (!(lower_bound >= kLowerBoundMin && lower_bound <= 0.0f)) return KDA_ERR_ARG;
    if (check_align) {
        for (const void* p : {q, k, v, g, static_cast<const void*>(out)})
            if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return KDA_ERR_ALIGN;
    }
    const size_t n_qk = (size_t)tok * H * kDim * 2, n_b = (size_t)tok * H * 2;
    for (const void* p : {q, k, v, g})
        if (overlaps(out, n_qk, p, n_qk)) return KDA_ERR_ALIAS;
    if (overlaps(out, n_qk, beta, n_b)) return KDA_ERR_ALIAS;
    const int N = cu ? num_seqs : B;
    const size_t ns = (size_t)N * H * kDim * kDim;
    if (s0 && s1) {
        const size_t b0 = ns * (s0_dtype == KDA_F32 ? 4 : 2), b1 = ns * (s1_dtype == KDA_F32 ? 4 : 2);
        if (overlaps(s0, b0, s1, b1) && (s0 != s1 || s0_dtype != s1_dtype)) return KDA_ERR_ALIAS;
    }
    if (s1 && overlaps(out, n_qk, s1, ns * (s1_dtype == KDA_F32 ? 4 : 2))) return KDA_ERR_ALIAS;
    return KDA_OK;
}

// Host-side checks of kda_bwd; no CUDA call.
int validate_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                 float scale, const float* A_log, const float* dt_bias, float lower_bound,
                 const void* s0, int s0_dtype, const void* dout, const float* dfinal,
                 const float* const* outs, const float* d_init, const int32_t* cu, int num_seqs,
                 int B, int T, int H, int K, int V) {
    if (K != kDim || V != kDim) return KDA_ERR_UNSUPPORTED_DIM;
    if (B < 1 || T < 0 || H < 1) return KDA_ERR_SHAPE;
    if (cu && (B != 1 || num_seqs < 1)) return KDA_ERR_SHAPE;
    const long long tok = (long long)B * T;
    if (tok * H * kDim >= (1LL << 31)) return KDA_ERR_SHAPE;
    const int N = cu ? num_seqs : B;
    if ((long long)N * H * kDim * kDim >= (1LL << 40)) return KDA_ERR_SHAPE;
    if (!A_log || !dt_bias || !outs[5] || !outs[6]) return KDA_ERR_NULL;   // dA_log, ddt_bias
    if (tok > 0) {
        if (!q || !k || !v || !g || !beta || !dout) return KDA_ERR_NULL;
        for (int i = 0; i < 5; ++i)
            if (!outs[i]) return KDA_ERR_NULL;
    }
    if (s0 && s0_dtype != KDA_BF16 && s0_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!std::isfinite(scale)) return KDA_ERR_ARG;
    if (!(lower_bound >= kLowerBoundMin && lower_bound <= 0.0f)) return KDA_ERR_ARG;
    for (const void* p : {q, k, v, g, dout, static_cast<const void*>(outs[2]),
                          static_cast<const void*>(d_init)})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return KDA_ERR_ALIGN;
    // outputs (fp32) must not overlap the inputs or each other
    const size_t n_row = (size_t)tok * H * kDim, n_s = (size_t)N * H * kDim * kDim;
    const void* in_p[] = {q, k, v, g, dout, beta, s0, dfinal, A_log, dt_bias};
    const size_t in_n[] = {n_row * 2, n_row * 2, n_row * 2, n_row * 2, n_row * 2,
                           (size_t)tok * H * 2, n_s * (s0_dtype == KDA_F32 ? 4 : 2), n_s * 4,
                           (size_t)H * 4, (size_t)H * kDim * 4};
    const void* out_p[] = {outs[0], outs[1], outs[2], outs[3], outs[4], outs[5], outs[6], d_init};
    const size_t out_n[] = {n_row * 4, n_row * 4, n_row * 4, n_row * 4, (size_t)tok * H * 4,
                            (size_t)H * 4, (size_t)H * kDim * 4, n_s * 4};
    for (int o = 0; o < 8; ++o) {
        for (int i = 0; i < 10; ++i)
            if (overlaps(out_p[o], out_n[o], in_p[i], in_n[i])) return KDA_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 8; ++o2)
            if (overlaps(out_p[o], out_n[o], out_p[o2], out_n[o2])) return KDA_ERR_ALIAS;
    }
    return KDA_OK;
}

// Host-side checks of kda_decode; no CUDA call.
int validate_decode(const void* q, const void* k, const void* v, const void* g, const void* beta,
                    float scale, const void* out, const float* A_log, const float* dt_bias,
                    float lower_bound, const void* s0, int s0_dtype, const void* s1, int s1_dtype,
                    int N, int H, int K, int V) {
    if (K != kDim || V != kDim) return KDA_ERR_UNSUPPORTED_DIM;
    if (N < 0 || H < 1) return KDA_ERR_SHAPE;
    if ((long long)N * H >= (1LL << 31) || (long long)N * H * kDim * kDim >= (1LL << 40))
        return KDA_ERR_SHAPE;
    if (N > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (!A_log || !dt_bias) return KDA_ERR_NULL;
    if (s0 && s0_dtype != KDA_BF16 && s0_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (s1 && s1_dtype != KDA_BF16 && s1_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (!std::isfinite(scale)) return KDA_ERR_ARG;
    if (!(lower_bound >= kLowerBoundMin && lower_bound <= 0.0f)) return KDA_ERR_ARG;
    for (const void* p : {q, k, v, g, static_cast<const void*>(out), s0, static_cast<const void*>(s1)})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return KDA_ERR_ALIGN;
    const size_t n_row = (size_t)N * H * kDim * 2, n_b = (size_t)N * H * 2;
    for (const void* p : {q, k, v, g})
        if (overlaps(out, n_row, p, n_row)) return KDA_ERR_ALIAS;
    if (overlaps(out, n_row, beta, n_b)) return KDA_ERR_ALIAS;
    const size_t ns = (size_t)N * H * kDim * kDim;
    if (s0 && s1) {
        const size_t b0 = ns * (s0_dtype == KDA_F32 ? 4 : 2), b1 = ns * (s1_dtype == KDA_F32 ? 4 : 2);
        if (overlaps(s0, b0, s1, b1) && (s0 != s1 || s0_dtype != s1_dtype)) return KDA_ERR_ALIAS;
    }
    if (s1 && overlaps(out, n_row, s1, ns * (s1_dtype == KDA_F32 ? 4 : 2))) return KDA_ERR_ALIAS;
    return KDA_OK;
}

}  // namespace
}  // namespace kda

// ---- scratch of kda_fwd_noalloc -------------------------------------------------
// The varlen sequence map of kda_fwd_noalloc lives in this fixed device array
// instead of memory from the allocator.  In host code the name only stands in
// for the device copy: its device address comes from cudaGetSymbolAddress,
// looked up once per device (with that device current) and cached.
static __device__ __align__(256) int g_noalloc_scratch[KDA_NOALLOC_MAX_SEQS + 1];

namespace {
int* g_noalloc_addr[kda::kMaxDevices] = {};
std::mutex g_noalloc_mu;

int noalloc_scratch(int dev, int** addr) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return kda::cuda_fail(KDA_ERR_CUDA, e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        g_noalloc_addr[dev] = static_cast<int*>(p);
    }
    *addr = g_noalloc_addr[dev];
    return KDA_OK;
}
}  // namespace

namespace kda {
namespace {

// ---- kda_fwd_host for one long fixed-length sequence ---------------------------
// The tokens are cut into blocks (multiples of the 16-token chunk, so that the
// chunking and every result are those of one kda_fwd call); block i runs while
// block i + 1 is copied in and block i - 1's output is copied out, on copy
// streams ordered against `s` by events.  The state passes from block to block
// through an fp32 device buffer (exact: the kernel keeps the state in fp32).
constexpr int kHostPipelineMin = 2048;   // tokens: shorter calls run in one block
constexpr int kHostBlockMin = 256;       // tokens: no block is halved below this

// First token of each block, then T.  Each block takes half of the tokens still left
// (rounded down to whole chunks) until that would be under kHostBlockMin: 4,096, 2,048,
// 1,024, 512, 256 and 256 tokens at T = 8,192.  The uploads run back to back whatever
// the split; what runs after the last one ends is the last block's kernel and download,
// so short blocks at the end finish sooner, and long ones at the start make fewer copies.
std::vector<int> host_blocks(int T) {
    std::vector<int> starts{0};
    for (int last = 0;;) {
        const int half = (T - last) / 2 / kChunk * kChunk;
        if (half < kHostBlockMin) break;
        last += half;
        starts.push_back(last);
    }
    starts.push_back(T);
    return starts;
}

bool host_pipelined(const int32_t* cu_seqlens, int B, int T) {
    return cu_seqlens == nullptr && B == 1 && T >= kHostPipelineMin;
}

int host_fwd_blocks(const void* q, const void* k, const void* v, const void* g, const void* beta,
                    float scale, void* out, const float* A_log, const float* dt_bias,
                    float lower_bound, const void* initial_state, int initial_state_dtype,
                    void* final_state, int final_state_dtype, int T, int H, cudaStream_t s) {
    const std::vector<int> starts = host_blocks(T);
    const int nblk = (int)starts.size() - 1;
    const size_t row = (size_t)H * kDim * 2, brow = (size_t)H * 2;   // bytes per token
    const size_t n_qk = (size_t)T * row, n_b = (size_t)T * brow;
    const size_t n_s = (size_t)H * kDim * kDim;
    const size_t b_s0 = initial_state ? n_s * (initial_state_dtype == KDA_F32 ? 4 : 2) : 0;
    const size_t b_s1 = final_state ? n_s * (final_state_dtype == KDA_F32 ? 4 : 2) : 0;
    // q, k, v, g, beta, out, A_log, dt_bias, initial, final, carried fp32 state
    const size_t sizes[] = {n_qk, n_qk, n_qk, n_qk, n_b, n_qk, sizeof(float) * H,
                            sizeof(float) * H * kDim, b_s0, b_s1, n_s * 4};
    size_t total = 0, offs[11];
    for (int i = 0; i < 11; ++i) {
        offs[i] = total;
        total += align_up(sizes[i]);
    }
    unsigned char* d = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d), total, s);
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_ALLOC, e);
    cudaStream_t sin = nullptr, sout = nullptr;
    std::vector<cudaEvent_t> ev(2 * nblk + 2, nullptr);   // in[i], kernel[i], alloc, out
    int rc = KDA_OK;
    e = cudaStreamCreateWithFlags(&sin, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&sout, cudaStreamNonBlocking);
    for (size_t i = 0; i < ev.size() && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    cudaEvent_t ev_alloc = ev[2 * nblk], ev_out = ev[2 * nblk + 1];
    // copies in: parameters and initial state, then the blocks back to back
    if (e == cudaSuccess) e = cudaEventRecord(ev_alloc, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sin, ev_alloc, 0);
    const void* params[] = {A_log, dt_bias, initial_state};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        if (params[i] && sizes[6 + i])
            e = cudaMemcpyAsync(d + offs[6 + i], params[i], sizes[6 + i], cudaMemcpyHostToDevice, sin);
    const void* tok_src[] = {q, k, v, g};
    for (int b = 0; b < nblk && e == cudaSuccess; ++b) {
        const size_t t0 = (size_t)starts[b], len = (size_t)(starts[b + 1] - starts[b]);
        for (int i = 0; i < 4 && e == cudaSuccess; ++i)
            e = cudaMemcpyAsync(d + offs[i] + t0 * row, static_cast<const unsigned char*>(tok_src[i]) + t0 * row,
                                len * row, cudaMemcpyHostToDevice, sin);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d + offs[4] + t0 * brow, static_cast<const unsigned char*>(beta) + t0 * brow,
                                len * brow, cudaMemcpyHostToDevice, sin);
        if (e == cudaSuccess) e = cudaEventRecord(ev[b], sin);
    }
    // blocks in order on `s`, each output block copied out as soon as it is written
    void* carry = d + offs[10];
    for (int b = 0; b < nblk && e == cudaSuccess && rc == KDA_OK; ++b) {
        const size_t t0 = (size_t)starts[b];
        const int len = starts[b + 1] - starts[b];
        const bool first = b == 0, last = b == nblk - 1;
        e = cudaStreamWaitEvent(s, ev[b], 0);
        if (e != cudaSuccess) break;
        // one pass per block (num_segments = 1): the blocks follow one another, so the
        // result is that of one one-pass call on all the tokens
        rc = kda_fwd_segments(
            d + offs[0] + t0 * row, d + offs[1] + t0 * row, d + offs[2] + t0 * row,
            d + offs[3] + t0 * row, d + offs[4] + t0 * brow, scale, d + offs[5] + t0 * row,
            reinterpret_cast<const float*>(d + offs[6]), reinterpret_cast<const float*>(d + offs[7]),
            lower_bound, first ? (initial_state ? static_cast<void*>(d + offs[8]) : nullptr) : carry,
            first ? initial_state_dtype : KDA_F32,
            last ? (final_state ? static_cast<void*>(d + offs[9]) : nullptr) : carry,
            last ? final_state_dtype : KDA_F32, nullptr, 0, 1, len, H, kDim, kDim, 1, s);
        if (rc != KDA_OK) break;
        e = cudaEventRecord(ev[nblk + b], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sout, ev[nblk + b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<unsigned char*>(out) + t0 * row, d + offs[5] + t0 * row,
                                (size_t)len * row, cudaMemcpyDeviceToHost, sout);
        if (e == cudaSuccess && last && final_state)
            e = cudaMemcpyAsync(final_state, d + offs[9], b_s1, cudaMemcpyDeviceToHost, sout);
    }
    // `s` takes over the copy streams' work before the buffer is freed
    if (sin) {
        const cudaError_t e1 = cudaEventRecord(ev_alloc, sin);
        if (e1 == cudaSuccess) cudaStreamWaitEvent(s, ev_alloc, 0);
    }
    if (sout) {
        const cudaError_t e1 = cudaEventRecord(ev_out, sout);
        if (e1 == cudaSuccess) cudaStreamWaitEvent(s, ev_out, 0);
    }
    cudaFreeAsync(d, s);
    const cudaError_t es = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = es;
    for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
    if (sin) cudaStreamDestroy(sin);
    if (sout) cudaStreamDestroy(sout);
    if (rc != KDA_OK) return rc;
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_NULL: return "KDA_ERR_NULL: a required pointer is NULL";
        case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE: inconsistent or out-of-range sizes";
        case KDA_ERR_UNSUPPORTED_DIM: return "KDA_ERR_UNSUPPORTED_DIM: only K = V = 128";
        case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN: q, k, v, g and out must be 16-byte aligned";
        case KDA_ERR_DTYPE: return "KDA_ERR_DTYPE: state dtype must be KDA_BF16 or KDA_F32";
        case KDA_ERR_LAUNCH: return "KDA_ERR_LAUNCH: kernel launch failed";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
        case KDA_ERR_BAD_SEQLENS: return "KDA_ERR_BAD_SEQLENS: cu_seqlens must rise from 0 to T";
        case KDA_ERR_ARCH: return "KDA_ERR_ARCH: needs a compute capability 10.3 (sm_103) GPU";
        case KDA_ERR_ALLOC: return "KDA_ERR_ALLOC: scratch allocation failed";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
        case KDA_ERR_ARG: return "KDA_ERR_ARG: scale must be finite, lower_bound in [-5.4, 0]";
        case KDA_ERR_ALIAS: return "KDA_ERR_ALIAS: out overlaps an input or states alias unsafely";
        case KDA_ERR_SEGMENTS:
            return "KDA_ERR_SEGMENTS: num_segments must be 0 (automatic), 1, or at most the "
                   "number of 16-token chunks of a fixed-length call";
        case KDA_ERR_SCRATCH_LIMIT:
            return "KDA_ERR_SCRATCH_LIMIT: kda_fwd_noalloc takes at most KDA_NOALLOC_MAX_SEQS "
                   "(65536) sequences";
        default: return "unknown kda_status";
    }
}

size_t kda_fwd_workspace_bytes(int B, int T, int H, int num_seqs, int varlen) {
    if (B < 1 || T < 0 || H < 1) return 0;
    if (varlen) return scratch_bytes(num_seqs, true);
    // a fixed-length call that kda_fwd splits into segments on the current device
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int segs = plan_segments(B, T, H, 0, sms);
    return segs >= 2 ? split_bytes(B, H, segs) : 0;
}

int kda_fwd_segments(const void* q, const void* k, const void* v, const void* g, const void* beta,
                     float scale, void* out, const float* A_log, const float* dt_bias,
                     float lower_bound, const void* initial_state, int initial_state_dtype,
                     void* final_state, int final_state_dtype, const int32_t* cu_seqlens,
                     int num_seqs, int B, int T, int H, int K, int V, int num_segments,
                     void* stream) {
    int rc = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                      initial_state_dtype, final_state, final_state_dtype, cu_seqlens, num_seqs,
                      B, T, H, K, V, true);
    if (rc != KDA_OK) return rc;
    const bool varlen = cu_seqlens != nullptr;
    if (num_segments < 0 || (varlen && num_segments > 1)) return KDA_ERR_SEGMENTS;
    if (!varlen && num_segments >= 2 && plan_segments(B, T, H, num_segments, 0) == 0)
        return KDA_ERR_SEGMENTS;
    int dev = 0, sms = 0;
    int* err = nullptr;
    rc = device_setup(&dev, &err, &sms);
    if (rc != KDA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int N = varlen ? num_seqs : B;
    const int segs = varlen ? 1 : plan_segments(B, T, H, num_segments, sms);
    if (segs == 0) return KDA_ERR_SEGMENTS;
    const size_t bytes = segs >= 2 ? split_bytes(N, H, segs) : scratch_bytes(N, varlen);

    unsigned char* scratch = nullptr;
    if (bytes > 0) {
        const cudaError_t ea = cudaMallocAsync(reinterpret_cast<void**>(&scratch), bytes, s);
        if (ea != cudaSuccess) return cuda_fail(KDA_ERR_ALLOC, ea);
    }
    Problem P;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.k = static_cast<const __nv_bfloat16*>(k);
    P.v = static_cast<const __nv_bfloat16*>(v);
    P.g = static_cast<const __nv_bfloat16*>(g);
    P.beta = static_cast<const __nv_bfloat16*>(beta);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.scale = scale;
    P.lower_bound = lower_bound;
    P.init_state = initial_state;
    P.init_dtype = initial_state_dtype;
    P.final_state = final_state;
    P.final_dtype = final_state_dtype;
    P.cu_seqlens = cu_seqlens;
    P.N = N;
    P.T = T;
    P.H = H;

    SeqMap M{};
    cudaError_t e = cudaSuccess;
    if (segs >= 2) {
        // initial states -> window 0 -> combine -> window 1 -> final state, all on the
        // caller's stream; every unit's states live at its own index of fp32 scratch
        const SplitScratch L = split_layout(N, H, segs);
        float* init0 = reinterpret_cast<float*>(scratch + L.init0);
        float* end0 = reinterpret_cast<float*>(scratch + L.end0);
        float* init1 = reinterpret_cast<float*>(scratch + L.init1);
        float* end1 = init0;   // free once window 0 has run
        auto* zero = reinterpret_cast<__nv_bfloat16*>(scratch + L.zero);
        Problem P0 = P, P1 = P;
        P0.window = 0;
        P0.nseg = segs;
        P0.vzero = zero;
        P0.init_state = init0;
        P0.init_dtype = KDA_F32;
        P0.final_state = end0;
        P0.final_dtype = KDA_F32;
        P1.window = 1;
        P1.nseg = segs;
        P1.init_state = init1;
        P1.init_dtype = KDA_F32;
        P1.final_state = end1;
        P1.final_dtype = KDA_F32;
        e = cudaMemsetAsync(zero, 0, (size_t)kChunk * H * kDim * 2, s);
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_SEGPREP, s, [&] {
                return launch_segprep(initial_state, initial_state_dtype, init0, N, H, segs, s);
            });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_FUSED, s, [&] { return launch_fused(P0, M, err, s); });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_COMBINE, s,
                             [&] { return launch_combine(end0, init1, N, H, segs, s); });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_FUSED, s, [&] { return launch_fused(P1, M, err, s); });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_SEGFINAL, s, [&] {
                return launch_segfinal(end1, final_state, final_state_dtype, N, H, segs, s);
            });
    } else {
        if (varlen) {
            M.seq_order = reinterpret_cast<int*>(scratch);
            M.valid = M.seq_order + N;
            // short sequences: persistent CTAs (when there are more units than SMs)
            if ((long long)T <= (long long)kPersistMaxAvgTokens * N) M.counter = M.seq_order + N + 1;
            e = timed_launch(KDA_KERNEL_SEQMAP, s, [&] { return launch_seqmap(P, M, err, s); });
        }
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_FUSED, s, [&] { return launch_fused(P, M, err, s); });
    }
    if (scratch) cudaFreeAsync(scratch, s);
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_LAUNCH, e);
    return KDA_OK;
}

int kda_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
            float scale, void* out, const float* A_log, const float* dt_bias, float lower_bound,
            const void* initial_state, int initial_state_dtype, void* final_state,
            int final_state_dtype, const int32_t* cu_seqlens, int num_seqs, int B, int T, int H,
            int K, int V, void* stream) {
    return kda_fwd_segments(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                            initial_state, initial_state_dtype, final_state, final_state_dtype,
                            cu_seqlens, num_seqs, B, T, H, K, V, 0, stream);
}

int kda_fwd_get_error(void* stream) {
    int dev = 0;
    int* err = nullptr;
    int rc = device_setup(&dev, &err);
    if (rc == KDA_ERR_CUDA) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    return word;
}

int kda_fwd_host(const void* q, const void* k, const void* v, const void* g, const void* beta,
                 float scale, void* out, const float* A_log, const float* dt_bias,
                 float lower_bound, const void* initial_state, int initial_state_dtype,
                 void* final_state, int final_state_dtype, const int32_t* cu_seqlens, int num_seqs,
                 int B, int T, int H, int K, int V, void* stream) {
    int rc = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                      initial_state_dtype, final_state, final_state_dtype, cu_seqlens, num_seqs,
                      B, T, H, K, V, false);
    if (rc != KDA_OK) return rc;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return KDA_ERR_BAD_SEQLENS;
        for (int n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_BAD_SEQLENS;
    }
    int dev = 0;
    int* err = nullptr;
    rc = device_setup(&dev, &err);
    if (rc != KDA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (host_pipelined(cu_seqlens, B, T))
        return host_fwd_blocks(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                               initial_state, initial_state_dtype, final_state, final_state_dtype,
                               T, H, s);
    const size_t tok = (size_t)B * T;
    const int N = cu_seqlens ? num_seqs : B;
    const size_t n_qk = tok * H * kDim * 2, n_b = tok * H * 2;
    const size_t n_s = (size_t)N * H * kDim * kDim;
    const size_t b_s0 = initial_state ? n_s * (initial_state_dtype == KDA_F32 ? 4 : 2) : 0;
    const size_t b_s1 = final_state ? n_s * (final_state_dtype == KDA_F32 ? 4 : 2) : 0;
    const size_t b_cu = cu_seqlens ? sizeof(int32_t) * (num_seqs + 1) : 0;
    const size_t sizes[] = {n_qk, n_qk, n_qk, n_qk, n_b, n_qk, sizeof(float) * H,
                            sizeof(float) * H * kDim, b_s0, b_s1, b_cu};
    size_t total = 0, offs[11];
    for (int i = 0; i < 11; ++i) {
        offs[i] = total;
        total += align_up(sizes[i]);
    }
    unsigned char* d = nullptr;
    const cudaError_t ea = cudaMallocAsync(reinterpret_cast<void**>(&d), total, s);
    if (ea != cudaSuccess) return cuda_fail(KDA_ERR_ALLOC, ea);
    const void* hsrc[] = {q, k, v, g, beta, nullptr, A_log, dt_bias, initial_state, nullptr,
                          cu_seqlens};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 11 && e == cudaSuccess; ++i)
        if (hsrc[i] && sizes[i])
            e = cudaMemcpyAsync(d + offs[i], hsrc[i], sizes[i], cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) {
        rc = kda_fwd(d + offs[0], d + offs[1], d + offs[2], d + offs[3], d + offs[4], scale,
                     d + offs[5], reinterpret_cast<const float*>(d + offs[6]),
                     reinterpret_cast<const float*>(d + offs[7]), lower_bound,
                     initial_state ? d + offs[8] : nullptr, initial_state_dtype,
                     final_state ? d + offs[9] : nullptr, final_state_dtype,
                     cu_seqlens ? reinterpret_cast<const int32_t*>(d + offs[10]) : nullptr,
                     num_seqs, B, T, H, K, V, stream);
        if (rc == KDA_OK && n_qk)
            e = cudaMemcpyAsync(out, d + offs[5], n_qk, cudaMemcpyDeviceToHost, s);
        if (rc == KDA_OK && e == cudaSuccess && final_state)
            e = cudaMemcpyAsync(final_state, d + offs[9], b_s1, cudaMemcpyDeviceToHost, s);
    }
    cudaFreeAsync(d, s);
    const cudaError_t es = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = es;
    if (rc != KDA_OK) return rc;
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_CUDA, e);
    return KDA_OK;
}

int kda_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                    const void* beta, float scale, void* out, const float* A_log,
                    const float* dt_bias, float lower_bound, const void* initial_state,
                    int initial_state_dtype, void* final_state, int final_state_dtype,
                    const int32_t* cu_seqlens, int num_seqs, int B, int T, int H, int K, int V,
                    void* stream) {
    int rc = validate(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                      initial_state_dtype, final_state, final_state_dtype, cu_seqlens, num_seqs,
                      B, T, H, K, V, true);
    if (rc != KDA_OK) return rc;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && num_seqs > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_SCRATCH_LIMIT;
    int dev = 0;
    int* err = nullptr;
    rc = device_setup(&dev, &err);
    if (rc != KDA_OK) return rc;
    int* scratch = nullptr;
    if (varlen) {
        rc = noalloc_scratch(dev, &scratch);
        if (rc != KDA_OK) return rc;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int N = varlen ? num_seqs : B;
    Problem P;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.k = static_cast<const __nv_bfloat16*>(k);
    P.v = static_cast<const __nv_bfloat16*>(v);
    P.g = static_cast<const __nv_bfloat16*>(g);
    P.beta = static_cast<const __nv_bfloat16*>(beta);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.scale = scale;
    P.lower_bound = lower_bound;
    P.init_state = initial_state;
    P.init_dtype = initial_state_dtype;
    P.final_state = final_state;
    P.final_dtype = final_state_dtype;
    P.cu_seqlens = cu_seqlens;
    P.N = N;
    P.T = T;
    P.H = H;
    SeqMap M{};
    if (varlen) {
        M.seq_order = scratch;       // every entry rewritten by the sequence map
        M.valid = scratch + N;       // set to 0 or 1 by the sequence map
    }
    cudaError_t e = cudaSuccess;
    if (varlen) e = timed_launch(KDA_KERNEL_SEQMAP, s, [&] { return launch_seqmap(P, M, err, s); });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_FUSED, s, [&] { return launch_fused(P, M, err, s); });
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_LAUNCH, e);
    return KDA_OK;
}

int kda_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
            float scale, const float* A_log, const float* dt_bias, float lower_bound,
            const void* initial_state, int initial_state_dtype, const void* d_out,
            const float* d_final_state, float* dq, float* dk, float* dv, float* dg, float* dbeta,
            float* dA_log, float* ddt_bias, float* d_initial_state, const int32_t* cu_seqlens,
            int num_seqs, int B, int T, int H, int K, int V, void* stream) {
    const float* outs[7] = {dq, dk, dv, dg, dbeta, dA_log, ddt_bias};
    int rc = validate_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state,
                          initial_state_dtype, d_out, d_final_state, outs, d_initial_state,
                          cu_seqlens, num_seqs, B, T, H, K, V);
    if (rc != KDA_OK) return rc;
    int dev = 0;
    int* err = nullptr;
    rc = device_setup(&dev, &err);
    if (rc != KDA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool varlen = cu_seqlens != nullptr;
    const int N = varlen ? num_seqs : B;
    const long long rows = (long long)B * T;
    size_t n_ck, n_fw, n_part, n_blk;
    const size_t floats = bwd_scratch_floats(N, rows, H, &n_ck, &n_fw, &n_part, &n_blk);
    const size_t map_bytes = scratch_bytes(N, varlen);
    unsigned char* scratch = nullptr;
    const cudaError_t ea = cudaMallocAsync(reinterpret_cast<void**>(&scratch),
                                           map_bytes + floats * sizeof(float), s);
    if (ea != cudaSuccess) return cuda_fail(KDA_ERR_ALLOC, ea);
    BwdProblem P{};
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.k = static_cast<const __nv_bfloat16*>(k);
    P.v = static_cast<const __nv_bfloat16*>(v);
    P.g = static_cast<const __nv_bfloat16*>(g);
    P.beta = static_cast<const __nv_bfloat16*>(beta);
    P.dout = static_cast<const __nv_bfloat16*>(d_out);
    P.scale = scale;
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.lower_bound = lower_bound;
    P.init_state = initial_state;
    P.init_dtype = initial_state_dtype;
    P.dfinal = d_final_state;
    P.dq = dq;
    P.dk = dk;
    P.dv = dv;
    P.dg = dg;
    P.dbeta = dbeta;
    P.dA_log = dA_log;
    P.ddt_bias = ddt_bias;
    P.d_init = d_initial_state;
    P.cu_seqlens = cu_seqlens;
    P.N = N;
    P.T = T;
    P.H = H;
    float* f = reinterpret_cast<float*>(scratch + map_bytes);
    P.ck = f;
    P.fw = f + n_ck;
    P.part = P.fw + n_fw;
    P.blk = P.part + n_part;
    cudaError_t e = cudaSuccess;
    const int* valid = nullptr;
    if (varlen) {   // validate cu_seqlens on the device (the sequence map's check)
        Problem FP{};
        FP.cu_seqlens = cu_seqlens;
        FP.N = N;
        FP.T = T;
        FP.H = H;
        SeqMap M{};
        M.seq_order = reinterpret_cast<int*>(scratch);
        M.valid = M.seq_order + N;
        valid = M.valid;
        e = timed_launch(KDA_KERNEL_SEQMAP, s, [&] { return launch_seqmap(FP, M, err, s); });
    }
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD, s, [&] { return launch_bwd_main(P, valid, s); });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_FINISH, s, [&] { return launch_bwd_finish(P, rows, valid, s); });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_REDUCE, s, [&] { return launch_bwd_reduce(P, rows, valid, s); });
    cudaFreeAsync(scratch, s);
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_LAUNCH, e);
    return KDA_OK;
}

size_t kda_bwd_workspace_bytes(int B, int T, int H, int num_seqs, int varlen) {
    if (B < 1 || T < 0 || H < 1) return 0;
    const int N = varlen ? num_seqs : B;
    size_t a, b, c, d;
    return scratch_bytes(N, varlen != 0) +
           bwd_scratch_floats(N, (long long)B * T, H, &a, &b, &c, &d) * sizeof(float);
}

int kda_decode(const void* q, const void* k, const void* v, const void* g, const void* beta,
               float scale, void* out, const float* A_log, const float* dt_bias, float lower_bound,
               const void* state_in, int state_in_dtype, void* state_out, int state_out_dtype,
               int N, int H, int K, int V, void* stream) {
    int rc = validate_decode(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, state_in,
                             state_in_dtype, state_out, state_out_dtype, N, H, K, V);
    if (rc != KDA_OK) return rc;
    int dev = 0;
    int* err = nullptr;
    rc = device_setup(&dev, &err);
    if (rc != KDA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem P{};
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.k = static_cast<const __nv_bfloat16*>(k);
    P.v = static_cast<const __nv_bfloat16*>(v);
    P.g = static_cast<const __nv_bfloat16*>(g);
    P.beta = static_cast<const __nv_bfloat16*>(beta);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.A_log = A_log;
    P.dt_bias = dt_bias;
    P.scale = scale;
    P.lower_bound = lower_bound;
    P.init_state = state_in;
    P.init_dtype = state_in_dtype;
    P.final_state = state_out;
    P.final_dtype = state_out_dtype;
    P.cu_seqlens = nullptr;
    P.N = N;
    P.T = 1;
    P.H = H;
    const cudaError_t e = timed_launch(KDA_KERNEL_DECODE, s, [&] { return launch_decode(P, s); });
    if (e != cudaSuccess) return cuda_fail(KDA_ERR_LAUNCH, e);
    return KDA_OK;
}

int kda_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (on) {
        for (auto& r : g_prof.pending) {
            cudaEventSynchronize(r.stop);
            g_prof.free_events.push_back(r.start);
            g_prof.free_events.push_back(r.stop);
        }
        g_prof.pending.clear();
        for (int i = 0; i < KDA_NUM_KERNELS; ++i) {
            g_prof.total_ms[i] = 0.0;
            g_prof.launches[i] = 0;
        }
    }
    g_prof.on = on != 0;
    return KDA_OK;
}

int kda_profile_read(double* total_ms, long long* launches) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    int rc = KDA_OK;
    for (auto& r : g_prof.pending) {
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) {
            rc = cuda_fail(KDA_ERR_CUDA, e);
        } else {
            g_prof.total_ms[r.kernel] += ms;
            g_prof.launches[r.kernel] += 1;
        }
        g_prof.free_events.push_back(r.start);
        g_prof.free_events.push_back(r.stop);
    }
    g_prof.pending.clear();
    for (int i = 0; i < KDA_NUM_KERNELS; ++i) {
        if (total_ms) total_ms[i] = g_prof.total_ms[i];
        if (launches) launches[i] = g_prof.launches[i];
    }
    return rc;
}

int kda_last_cuda_error(void) { return t_last_cuda_error; }

const char* kda_kernel_name(int kernel_id) {
    switch (kernel_id) {
        case KDA_KERNEL_SEQMAP: return "seqmap_kernel";
        case KDA_KERNEL_FUSED: return "fused_kernel";
        case KDA_KERNEL_DECODE: return "decode_kernel";
        case KDA_KERNEL_COMBINE: return "combine_kernel";
        case KDA_KERNEL_SEGPREP: return "segprep_kernel";
        case KDA_KERNEL_SEGFINAL: return "segfinal_kernel";
        case KDA_KERNEL_BWD: return "bwd_kernel";
        case KDA_KERNEL_BWD_FINISH: return "bwd_finish_kernel";
        case KDA_KERNEL_BWD_REDUCE: return "bwd_reduce_kernel";
        default: return "unknown";
    }
}

}  // extern "C"
