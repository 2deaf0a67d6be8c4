// Variable-length chunk map (one CTA): validates cu_seqlens on the device and
// builds, without any host synchronisation,
//   chunk_first[n]  first global 16-token chunk of sequence n (prefix sum of
//                   ceil(L_n / 16)); chunks never cross a sequence boundary
//   chunk_seq[j]    owning sequence of chunk j (-1 for unused slots)
//   seq_order[r]    sequences sorted by length, longest first, so that the
//                   state kernel starts the longest recurrences first
// Variable-length batching through cu_seqlens: "Moonshot AI Rilis FlashKDA"
// (captivela.com), paragraph on cu_seqlens.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;
constexpr int kSortMax = 4096;   // rank sort above this count falls back to input order

__global__ void __launch_bounds__(kThreads) chunkmap_kernel(Problem P, ChunkMap M, int* err) {
    __shared__ int bad;
    __shared__ int carry;
    __shared__ int scan[kThreads];
    const int N = P.N;
    const int* cu = P.cu_seqlens;
    if (threadIdx.x == 0) {
        bad = (cu[0] != 0) || (cu[N] != P.T);
        carry = 0;
    }
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += kThreads)
        if (cu[n + 1] < cu[n]) bad = 1;
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) {
            *M.valid = 0;
            set_error(err, KDA_ERR_BAD_SEQLENS);
        }
        for (int j = threadIdx.x; j < P.chunk_bound; j += kThreads) M.chunk_seq[j] = -1;
        return;
    }
    // prefix sum of chunk counts, kThreads sequences per tile
    for (int base = 0; base < N; base += kThreads) {
        int n = base + threadIdx.x;
        int c = n < N ? (cu[n + 1] - cu[n] + kChunk - 1) / kChunk : 0;
        scan[threadIdx.x] = c;
        __syncthreads();
        for (int off = 1; off < kThreads; off <<= 1) {
            int x = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
            __syncthreads();
            scan[threadIdx.x] += x;
            __syncthreads();
        }
        if (n < N) M.chunk_first[n] = carry + scan[threadIdx.x] - c;
        __syncthreads();
        if (threadIdx.x == kThreads - 1) carry += scan[kThreads - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) M.chunk_first[N] = carry;
    __syncthreads();
    const int total = carry;
    for (int n = threadIdx.x; n < N; n += kThreads) {
        int j0 = M.chunk_first[n], j1 = M.chunk_first[n + 1];
        for (int j = j0; j < j1; ++j) M.chunk_seq[j] = n;
    }
    for (int j = total + threadIdx.x; j < P.chunk_bound; j += kThreads) M.chunk_seq[j] = -1;
    // longest-first order (stable rank sort; input order above kSortMax)
    for (int n = threadIdx.x; n < N; n += kThreads) {
        if (N > kSortMax) {
            M.seq_order[n] = n;
            continue;
        }
        int Ln = cu[n + 1] - cu[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            int Lm = cu[m + 1] - cu[m];
            rank += (Lm > Ln) || (Lm == Ln && m < n);
        }
        M.seq_order[rank] = n;
    }
    if (threadIdx.x == 0) *M.valid = 1;
}

}  // namespace

cudaError_t launch_chunkmap(const Problem& P, const ChunkMap& M, int* err, cudaStream_t s) {
    chunkmap_kernel<<<1, kThreads, 0, s>>>(P, M, err);
    return cudaGetLastError();
}

}  // namespace kda
