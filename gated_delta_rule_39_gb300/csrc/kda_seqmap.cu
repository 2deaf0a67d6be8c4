// Variable-length sequence map (one CTA): validates cu_seqlens on the device
// and orders the sequences longest first, so that the fused kernel starts
// the longest recurrences first; no host synchronisation.
// Variable-length batching through cu_seqlens: "Moonshot AI Rilis FlashKDA"
// (captivela.com), paragraph on cu_seqlens.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;
constexpr int kSortMax = 8192;   // above this many sequences the input order is kept

__global__ void __launch_bounds__(kThreads) seqmap_kernel(Problem P, SeqMap M, int* err) {
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
    // longest first (stable rank sort); input order above kSortMax sequences
    for (int n = threadIdx.x; n < N; n += kThreads) {
        if (N > kSortMax) {
            M.seq_order[n] = n;
            continue;
        }
        const int Ln = cu[n + 1] - cu[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int Lm = cu[m + 1] - cu[m];
            rank += (Lm > Ln) || (Lm == Ln && m < n);
        }
        M.seq_order[rank] = n;
    }
    if (threadIdx.x == 0) *M.valid = 1;
}

}  // namespace

cudaError_t launch_seqmap(const Problem& P, const SeqMap& M, int* err, cudaStream_t s) {
    seqmap_kernel<<<1, kThreads, 0, s>>>(P, M, err);
    return cudaGetLastError();
}

}  // namespace kda
