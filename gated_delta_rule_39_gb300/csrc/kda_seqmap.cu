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
constexpr int kWarps = kThreads / 32;
constexpr int kSortMax = 16384;   // up to this many sequences: exact longest-first order
constexpr size_t kSortSmem = sizeof(unsigned long long) * kSortMax;   // 128 KB
constexpr int kBuckets = 32;      // above it: order by floor(log2(length + 1)), descending

// Up to kSortMax sequences the order is a bitonic sort of the keys
// (max - length) << 32 | index in shared memory: longest first, ties in input order
// (a stable order without a stable sort).  Above it, a stable counting sort by the
// length's binary order of magnitude (longest bucket first, input order inside a
// bucket): warp w owns a contiguous segment of the sequences, counts its buckets,
// a scan over (bucket descending, warp) gives each warp's first slot per bucket, and
// each warp places its segment in input order.  Both orders only decide which
// (sequence, head) units start first; every unit's result is independent of them.
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
        int* cnt = reinterpret_cast<int*>(keys);   // [kWarps][kBuckets] counts, then first slots
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int per = (N + kWarps - 1) / kWarps;
        const int n0 = min(N, w * per), n1 = min(N, n0 + per);
        const auto bucket = [&](int n) {   // floor(log2(length + 1)), 0 .. 31
            return 31 - __clz((unsigned)(cu[n + 1] - cu[n]) + 1u);
        };
        if (lane < kBuckets) cnt[w * kBuckets + lane] = 0;
        __syncwarp();
        for (int base = n0; base < n1; base += 32) {
            const int n = base + lane;
            const bool in = n < n1;
            const int b = in ? bucket(n) : -1 - lane;   // distinct dummies outside the segment
            const unsigned same = __match_any_sync(0xffffffffu, b);
            if (in && lane == __ffs(same) - 1) cnt[w * kBuckets + b] += __popc(same);
            __syncwarp();
        }
        __syncthreads();
        // exclusive scan in the order (bucket descending, warp ascending): thread
        // i = (kBuckets - 1 - b) * kWarps + w holds the count of (w, b)
        {
            const int i = threadIdx.x;
            const int b = kBuckets - 1 - i / kWarps, ww = i % kWarps;
            const int c = cnt[ww * kBuckets + b];
            int x = c;   // inclusive scan within the warp, then over warps
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            __shared__ int warp_tot[kWarps];
            if (lane == 31) warp_tot[w] = x;
            __syncthreads();
            if (w == 0) {
                int t = warp_tot[lane];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, t, d);
                    if (lane >= d) t += y;
                }
                warp_tot[lane] = t - warp_tot[lane];   // exclusive
            }
            __syncthreads();
            cnt[ww * kBuckets + b] = warp_tot[w] + x - c;   // first slot of (ww, b)
        }
        __syncthreads();
        for (int base = n0; base < n1; base += 32) {
            const int n = base + lane;
            const bool in = n < n1;
            const int b = in ? bucket(n) : -1 - lane;
            const unsigned same = __match_any_sync(0xffffffffu, b);
            if (in) {
                const int rank = __popc(same & ((1u << lane) - 1u));
                M.seq_order[cnt[w * kBuckets + b] + rank] = n;
            }
            __syncwarp();
            if (in && lane == __ffs(same) - 1) cnt[w * kBuckets + b] += __popc(same);
            __syncwarp();
        }
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
    if (threadIdx.x == 0) {
        *M.valid = 1;
        if (M.counter) *M.counter = 0;   // the fused kernel's persistent CTAs count from 0
    }
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
    // shared memory for the keys, or for the bucket counts of the counting sort
    const size_t smem = P.N <= kSortMax ? kSortSmem : sizeof(int) * kWarps * kBuckets;
    seqmap_kernel<<<1, kThreads, smem, s>>>(P, M, err);
    return cudaGetLastError();
}

}  // namespace kda
