// Internal definitions shared by the KDA forward kernels (sm_103a).
//
// Numerics (what each value is stored as, and why):
//   - gates, cumulative log-decays and their powers of two: fp32
//   - decay-ratio products A_kk = diag(b) (K*2^G)(K*2^-G)^T and
//     A_qk = (Q*2^G)(K*2^-G)^T: tf32 tensor-core MMA with fp32 accumulate.
//     2^-G reaches 2^115 inside a 16-token chunk, which needs an 8-bit
//     exponent, and the 10-bit tf32 mantissa keeps these products accurate.
//   - the sequential state recurrence runs on tcgen05 tensor cores with the
//     state S and U = u - w S held in tensor memory as fp32 and read directly
//     as the A operand of kind::tf32 MMAs; their partners (w, Q*2^G,
//     K*2^(G_C-G), A_qk) are fp32 rounded to tf32 (half away from zero).
//   - u = T diag(b) V: fp16 operands (V is bf16 data; the WY inverse's inputs
//     lie in [-1, 1], "Moonshot AI Open-Sources FlashKDA", "What makes the
//     kernel fast": fp16 16x16 inversion), fp32 accumulate.  w = T diag(b)
//     (K*2^G) likewise, with fp32 accumulate and a tf32 result.
//   - the recurrent state itself: fp32 accumulators.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kDim = 128;       // K = V
constexpr int kChunk = 16;      // tokens per chunk ("What makes the kernel fast": chunk 16)
constexpr float kLog2e = 1.4426950408889634f;

// ---- problem description shared by all kernels ------------------------------
struct Problem {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    __nv_bfloat16* out;
    const float* A_log;
    const float* dt_bias;
    float scale;
    float lower_bound;
    const void* init_state;
    int init_dtype;
    void* final_state;
    int final_dtype;
    const int* cu_seqlens;   // device, or nullptr for fixed length
    int N;                   // sequences
    int T;                   // tokens per sequence (fixed) or total tokens (varlen)
    int H;
    // Sequence split of fixed-length calls (window >= 0; see kda_split.cu).  Every
    // sequence's n = ceil(T / 16) chunks are cut into nseg segments: segment j holds
    // chunks floor(j n / nseg) .. floor((j + 1) n / nseg) - 1.  Unit `rank` of a window
    // reads its initial state and writes its final state at index rank (fp32).
    //   window 0: 2 nseg - 3 units per sequence: segment 0, then for each middle
    //             segment j its affine part and its transition operator (whose values
    //             are zero: v is read from the 16 zero rows at `vzero`).
    //   window 1: segments 1 .. nseg-1.
    // Every unit writes its outputs; those of window 0's middle units are overwritten
    // by window 1.
    int window = -1;         // -1: one unit per (sequence, head), no split
    int nseg = 0;
    const __nv_bfloat16* vzero = nullptr;   // [16][H][128] zeros (window 0)
};

// ---- backward pass (kda_bwd.cu) ----------------------------------------------------
struct BwdProblem {
    const __nv_bfloat16 *q, *k, *v, *g, *beta, *dout;
    float scale;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    const void* init_state;   // or nullptr (zero)
    int init_dtype;
    const float* dfinal;      // dL/d(final state) [N][H][K][V], or nullptr (zero)
    float *dq, *dk, *dv, *dg, *dbeta, *dA_log, *ddt_bias;
    float* d_init;            // dL/d(initial state) [N][H][K][V], or nullptr (not written)
    const int* cu_seqlens;    // or nullptr: N sequences of T tokens
    int N, T, H;
    float *ck, *fw, *part, *blk;   // scratch (bwd_scratch_floats)
};

// TMA tensor maps over the token rows of q, k, v, g (built on the host per call).
struct RawMaps {
    CUtensorMap q, k, v, g;
    CUtensorMap vz;   // zero rows (sequence split, window 0)
};

// Scratch written by the varlen sequence map, read by the fused kernel.
struct SeqMap {
    int* seq_order;     // [N] sequences, longest first
    int* valid;         // [1] 1 if cu_seqlens passed validation
    int* counter = nullptr;   // [1] next unit of a persistent launch (zeroed by the map)
};

// Device error word helpers.
__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// sigmoid(x) = 1 / (1 + 2^(-x log2 e))
__device__ __forceinline__ float sigmoid_fast(float x) {
    return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A(16x8 tf32, row) * B(8x8 tf32, col), fp32 accumulate
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_seqmap(const Problem& P, const SeqMap& M, int* err, cudaStream_t s);
cudaError_t launch_fused(const Problem& P, const SeqMap& M, int* err, cudaStream_t s);
cudaError_t launch_decode(const Problem& P, cudaStream_t s);
cudaError_t launch_combine(const float* w0, float* sin, int N, int H, int nseg, cudaStream_t s);
cudaError_t launch_segprep(const void* init, int init_dtype, float* w0init, int N, int H, int nseg,
                           cudaStream_t s);
cudaError_t launch_segfinal(const float* w1final, void* final_state, int final_dtype, int N, int H,
                            int nseg, cudaStream_t s);
size_t fused_smem_bytes();
size_t bwd_scratch_floats(int N, long long rows, int H, size_t* ck, size_t* fw, size_t* part,
                          size_t* blk);
cudaError_t launch_bwd_main(const BwdProblem& P, const int* valid, cudaStream_t s);
cudaError_t launch_bwd_finish(const BwdProblem& P, long long rows, const int* valid,
                              cudaStream_t s);
cudaError_t launch_bwd_reduce(const BwdProblem& P, long long rows, const int* valid,
                              cudaStream_t s);

}  // namespace kda
