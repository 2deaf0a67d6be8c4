// Sequence split of long fixed-length calls with few (sequence, head) units.
//
// The recurrence is affine in the state: over a segment j of a sequence, the
// chunkwise algorithm maps the state at the segment's start to the state at its
// end as  S_end = P_j S_start + B_j,  with P_j the product of the segment's
// per-token transitions (I - b_t k_t k_t^T) Diag(exp(gl_t)) and B_j the end
// state of the same segment run from a zero state.  So the segments of one
// sequence can run side by side in two windows:
//
//   window 0  segment 0 from the caller's initial state (its outputs are final);
//             for every middle segment j = 1 .. s-2, B_j (a run from a zero state)
//             and P_j (a run from the identity state with zero values: its end
//             state is P_j I = P_j);
//   combine   S_start(1) = end state of segment 0;
//             S_start(j) = P_{j-1} S_start(j-1) + B_{j-1},  j = 2 .. s-1;
//   window 1  segments 1 .. s-1 from S_start(j), writing their outputs; the last
//             one writes the caller's final state.
//
// That is 2s - 3 units per (sequence, head) in window 0 and s - 1 in window 1, each
// over a 1/s share of the tokens, so a call whose B*H units leave most SMs idle
// finishes in about 2/s of the one-pass time.  This is the chunk-parallel first
// stage of the pages' two-stage design carried one level up: the token-parallel
// work is spread over segments, and only the short combine step stays sequential
// ("Moonshot AI Open-Sources FlashKDA", "What makes the kernel fast": the
// sequential stage has far less parallelism than the token-parallel one).
//
// This file holds the steps around the two windows: the initial states of window 0
// (the caller's, zero, identity; fp32), the combine step (one CTA per (sequence,
// head), fp32 products of 128 x 128 matrices on CUDA cores, a chain of s - 2), and
// the copy of the last segment's end state into the caller's final state.  Each
// unit of a window reads and writes its states at its own index, so the fused
// kernel's epilogue is the same as for a one-pass call.
#include <atomic>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kCombThreads = 256;   // 16 x 16 threads, an 8 x 8 output tile each
constexpr int kPad = 132;           // row stride of the transposed operator (floats)
constexpr int kCopyThreads = 256;
constexpr size_t kKV = (size_t)kDim * kDim;   // elements of one state

struct CombSmem {
    float pt[kDim][kPad];   // P_{j-1} transposed: pt[k][r] = P[r][k]
    float s[kDim][kDim];    // S_start(j-1)
};

// w0: end states of window 0, [N][2s-3][H][128][128] fp32 (unit order of that window);
// sin: initial states of window 1, [N][s-1][H][128][128] fp32.
__global__ void __launch_bounds__(kCombThreads) combine_kernel(const float* __restrict__ w0,
                                                              float* __restrict__ sin, int H,
                                                              int nseg) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    CombSmem& S = *reinterpret_cast<CombSmem*>(smem_raw);
    const int h = blockIdx.x % H, seq = blockIdx.x / H;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int per0 = 2 * nseg - 3, per1 = nseg - 1;
    const auto w0_at = [&](int unit) { return w0 + ((size_t)(seq * per0 + unit) * H + h) * kKV; };
    const auto sin_at = [&](int j) { return sin + ((size_t)(seq * per1 + j - 1) * H + h) * kKV; };

    // S_start(1) = end state of segment 0 (window-0 unit 0)
    {
        const float4* src = reinterpret_cast<const float4*>(w0_at(0));
        float4* dst = reinterpret_cast<float4*>(sin_at(1));
        float4* sm = reinterpret_cast<float4*>(&S.s[0][0]);
        for (int i = tid; i < (int)(kKV / 4); i += kCombThreads) {
            const float4 x = src[i];
            dst[i] = x;
            sm[i] = x;
        }
    }
    for (int j = 2; j < nseg; ++j) {
        // P_{j-1}: window-0 unit s-2+(j-1); B_{j-1}: unit j-1
        const float* Pm = w0_at(nseg - 2 + (j - 1));
        const float* Bm = w0_at(j - 1);
        for (int i = tid; i < (int)kKV; i += kCombThreads) {
            const int r = i >> 7, k = i & 127;
            S.pt[k][r] = Pm[i];
        }
        __syncthreads();
        float acc[8][8];
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
        const int r0 = 8 * ty, c0 = 8 * tx;
#pragma unroll 4
        for (int k = 0; k < kDim; ++k) {
            const float4 p0 = *reinterpret_cast<const float4*>(&S.pt[k][r0]);
            const float4 p1 = *reinterpret_cast<const float4*>(&S.pt[k][r0 + 4]);
            const float4 s0 = *reinterpret_cast<const float4*>(&S.s[k][c0]);
            const float4 s1 = *reinterpret_cast<const float4*>(&S.s[k][c0 + 4]);
            const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(pr[a], sc[b], acc[a][b]);
        }
        __syncthreads();   // every thread has read S.s before it is overwritten
        float* dst = sin_at(j);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const size_t row = (size_t)(r0 + a) * kDim + c0;
            const float4 b0 = *reinterpret_cast<const float4*>(Bm + row);
            const float4 b1 = *reinterpret_cast<const float4*>(Bm + row + 4);
            const float4 o0 = make_float4(acc[a][0] + b0.x, acc[a][1] + b0.y, acc[a][2] + b0.z,
                                          acc[a][3] + b0.w);
            const float4 o1 = make_float4(acc[a][4] + b1.x, acc[a][5] + b1.y, acc[a][6] + b1.z,
                                          acc[a][7] + b1.w);
            *reinterpret_cast<float4*>(dst + row) = o0;
            *reinterpret_cast<float4*>(dst + row + 4) = o1;
            *reinterpret_cast<float4*>(&S.s[r0 + a][c0]) = o0;
            *reinterpret_cast<float4*>(&S.s[r0 + a][c0 + 4]) = o1;
        }
        __syncthreads();
    }
}

__device__ __forceinline__ float4 load4(const void* base, int dtype, size_t idx) {
    if (dtype == KDA_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + idx);
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}

// Window 0's initial states, unit rank = seq (2s - 3) + vj: vj = 0 the caller's state
// (zero without one), 1 .. s-2 zero (affine parts), s-1 .. 2s-4 identity (transition
// operators).  One CTA per (unit, head).
__global__ void __launch_bounds__(kCopyThreads) segprep_kernel(const void* __restrict__ init,
                                                              int init_dtype,
                                                              float* __restrict__ w0init, int H,
                                                              int nseg) {
    const int h = blockIdx.x % H, rank = blockIdx.x / H;
    const int per = 2 * nseg - 3, seq = rank / per, vj = rank % per;
    float4* dst = reinterpret_cast<float4*>(w0init + (size_t)blockIdx.x * kKV);
    const size_t src = ((size_t)seq * H + h) * kKV;
    for (int i = threadIdx.x; i < (int)(kKV / 4); i += kCopyThreads) {
        float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (vj == 0) {
            if (init) x = load4(init, init_dtype, src + 4 * (size_t)i);
        } else if (vj > nseg - 2) {
            const int r = (4 * i) >> 7, c = (4 * i) & 127;   // element (r, c .. c + 3)
            x.x = r == c ? 1.0f : 0.0f;
            x.y = r == c + 1 ? 1.0f : 0.0f;
            x.z = r == c + 2 ? 1.0f : 0.0f;
            x.w = r == c + 3 ? 1.0f : 0.0f;
        }
        dst[i] = x;
    }
}

// The caller's final state from window 1's last unit of each sequence.
__global__ void __launch_bounds__(kCopyThreads) segfinal_kernel(const float* __restrict__ w1final,
                                                               void* __restrict__ final_state,
                                                               int final_dtype, int H, int nseg) {
    const int h = blockIdx.x % H, seq = blockIdx.x / H;
    const int rank = seq * (nseg - 1) + nseg - 2;
    const float4* src = reinterpret_cast<const float4*>(w1final + ((size_t)rank * H + h) * kKV);
    const size_t dst = ((size_t)seq * H + h) * kKV;
    for (int i = threadIdx.x; i < (int)(kKV / 4); i += kCopyThreads) {
        const float4 x = src[i];
        if (final_dtype == KDA_F32) {
            reinterpret_cast<float4*>(static_cast<float*>(final_state) + dst)[i] = x;
        } else {
            const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y);
            const __nv_bfloat162 b = __floats2bfloat162_rn(x.z, x.w);
            uint2 raw;
            raw.x = *reinterpret_cast<const uint32_t*>(&a);
            raw.y = *reinterpret_cast<const uint32_t*>(&b);
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(final_state) + dst)[i] = raw;
        }
    }
}

}  // namespace

cudaError_t launch_segprep(const void* init, int init_dtype, float* w0init, int N, int H, int nseg,
                           cudaStream_t s) {
    const long long ctas = (long long)N * H * (2 * nseg - 3);
    if (ctas == 0) return cudaSuccess;
    segprep_kernel<<<(unsigned)ctas, kCopyThreads, 0, s>>>(init, init_dtype, w0init, H, nseg);
    return cudaGetLastError();
}

cudaError_t launch_segfinal(const float* w1final, void* final_state, int final_dtype, int N, int H,
                            int nseg, cudaStream_t s) {
    const long long ctas = (long long)N * H;
    if (ctas == 0 || final_state == nullptr) return cudaSuccess;
    segfinal_kernel<<<(unsigned)ctas, kCopyThreads, 0, s>>>(w1final, final_state, final_dtype, H,
                                                           nseg);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* w0, float* sin, int N, int H, int nseg, cudaStream_t s) {
    const long long ctas = (long long)N * H;
    if (ctas == 0 || nseg < 2) return cudaSuccess;
    const int smem = (int)sizeof(CombSmem);
    static std::atomic<bool> attr_set[64];   // per device; setting it twice is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
    }
    combine_kernel<<<(unsigned)ctas, kCombThreads, smem, s>>>(w0, sin, H, nseg);
    return cudaGetLastError();
}

}  // namespace kda
