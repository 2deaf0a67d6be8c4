// Variable-length sequence map (one CTA): validates cu_seqlens on the device
// and orders the sequences longest first, so that the fused kernel starts
// the longest recurrences first; no host synchronisation.
// Variable-length batching through cu_seqlens: "Moonshot AI Rilis FlashKDA"
// (captivela.com), paragraph on cu_seqlens.
#include <atomic>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;
constexpr int kSortMax = 16384;   // above this many sequences the input order is kept
constexpr size_t kSortSmem = sizeof(unsigned long long) * kSortMax;   // 128 KB

// The order is a bitonic sort of the keys (max - length) << 32 | index in shared
// memory: longest first, ties in input order (a stable order without a stable sort).
__global__ void __launch_bounds__(kThreads) seqmap_kernel(Problem P, SeqMap M, int* err) {
    extern __shared__ unsigned long long keys[];
    __shared__ int bad;
    const int N = P.N;
    const int* cu = P.cu_seqlens;
    if (threadIdx.x == 0) bad = (cu[0] != 0) || (cu[N] != P.T);
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += kThreads)
        if (cu[n + 1] < cu[n]) bad = 1;
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) {
            *M.valid = 0;
            set_error(err, KDA_ERR_BAD_SEQLENS);
        }
        return;
    }
    if (N > kSortMax) {
        for (int n = threadIdx.x; n < N; n += kThreads) M.seq_order[n] = n;
    } else {
        int n2 = 1;   // sorted length: a power of two, padded with keys that sort last
        while (n2 < N) n2 <<= 1;
        for (int i = threadIdx.x; i < n2; i += kThreads) {
            if (i < N) {
                const unsigned len = (unsigned)(cu[i + 1] - cu[i]);
                keys[i] = ((unsigned long long)(0x7FFFFFFFu - len) << 32) | (unsigned)i;
            } else {
                keys[i] = ~0ull;
            }
        }
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = threadIdx.x; i < n2; i += kThreads) {
                    const int p = i ^ j;
                    if (p > i) {
                        const unsigned long long a = keys[i], b = keys[p];
                        // ascending where bit k of i is clear, descending where it is set
                        if ((a > b) == ((i & k) == 0)) {
                            keys[i] = b;
                            keys[p] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
        for (int n = threadIdx.x; n < N; n += kThreads)
            M.seq_order[n] = (int)(keys[n] & 0xFFFFFFFFull);
    }
    if (threadIdx.x == 0) *M.valid = 1;
}

// per-device flag: the kernel attribute below is set once (setting it is idempotent,
// so two threads racing on a first call both succeed)
std::atomic<bool> g_attr_set[64];

}  // namespace

cudaError_t launch_seqmap(const Problem& P, const SeqMap& M, int* err, cudaStream_t s) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !g_attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(seqmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kSortSmem);
        if (e != cudaSuccess) return e;
        g_attr_set[dev].store(true, std::memory_order_release);
    }
    // shared memory for the keys only when there is something to sort
    const size_t smem = P.N <= kSortMax ? kSortSmem : 0;
    seqmap_kernel<<<1, kThreads, smem, s>>>(P, M, err);
    return cudaGetLastError();
}

}  // namespace kda
