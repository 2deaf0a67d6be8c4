// Inter-chunk state kernel: the sequential part of the chunked recurrence.
//
// One CTA per (sequence, head, 64-wide slice of value channels); value
// columns of the state evolve independently, so the slices never talk.  The
// state slice S[:, v0:v0+64] (fp32) lives in registers as the transposed
// tile S^T, 16 value rows per warp.  Per chunk, with intra-chunk factors
// qg, kd, w, u, A_qk, gc from the intra-chunk kernel:
//   U   = u - w S                         (16 x 64)
//   O   = scale ((Q*2^G) S + A_qk U)      (16 x 64, the chunk's outputs)
//   S  <- Diag(2^G_last) S + (K*2^(G_last-G))^T U
// computed in the transposed orientation (U^T = u^T - S^T w^T, ...) so that
// every accumulator tile feeds the next MMA as an A operand without a
// transpose.  Chunkwise DPLR-variant recurrence: "Moonshot AI Open-Sources
// FlashKDA", sections "Why KDA?" and "What makes the kernel fast" (a second,
// sequential stage after the token-parallel one).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kVS = 64;              // value channels per CTA
constexpr int kWarps = kVS / 16;     // 16 value rows of S^T per warp
constexpr int kStages = 4;           // chunks in flight (cp.async ring)
constexpr int LD = 136;              // fp16 per padded 128-wide row
constexpr int U_LD = 72;             // fp16 per padded 64-wide row
constexpr int AQ_LD = 24;            // fp16 per padded 16-wide row
constexpr int O_LD = 24;             // bf16 per padded row of the output staging tile

struct Stage {
    __half qg[kChunk * LD];
    __half kd[kChunk * LD];
    __half w[kChunk * LD];
    __half u[kChunk * U_LD];
    __half aqk[kChunk * AQ_LD];
    float gc[kDim];
};
static_assert(sizeof(Stage) % 16 == 0, "stage must stay 16-byte aligned");

struct Smem {
    Stage st[kStages];
    __nv_bfloat16 ostage[kWarps][kChunk * O_LD];
};

__device__ __forceinline__ void load_stage(Stage& st, const Workspace& W, size_t jh, int v0,
                                           int tid) {
    const __half* qg = W.qg + jh * (kChunk * kDim);
    const __half* kd = W.kd + jh * (kChunk * kDim);
    const __half* w = W.wneg + jh * (kChunk * kDim);
    const __half* u = W.u + jh * (kChunk * kDim);
    for (int i = tid; i < kChunk * 16; i += kWarps * 32) {
        const int r = i >> 4, p = i & 15;
        cp_async16(&st.qg[r * LD + p * 8], qg + r * kDim + p * 8);
        cp_async16(&st.kd[r * LD + p * 8], kd + r * kDim + p * 8);
        cp_async16(&st.w[r * LD + p * 8], w + r * kDim + p * 8);
    }
    for (int i = tid; i < kChunk * (kVS / 8); i += kWarps * 32) {
        const int r = i / (kVS / 8), p = i % (kVS / 8);
        cp_async16(&st.u[r * U_LD + p * 8], u + r * kDim + v0 + p * 8);
    }
    if (tid < 32) {
        const int r = tid >> 1, p = tid & 1;
        cp_async16(&st.aqk[r * AQ_LD + p * 8], W.aqk + jh * (kChunk * kChunk) + r * kChunk + p * 8);
    } else if (tid < 64) {
        const int p = tid - 32;
        cp_async16(&st.gc[p * 4], W.gc + jh * kDim + p * 4);
    }
}

__global__ void __launch_bounds__(kWarps * 32) state_kernel(Problem P, ChunkMap M, Workspace W) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int fg = lane >> 2, ft = lane & 3;
    constexpr int kSlices = kDim / kVS;
    int b = blockIdx.x;
    const int vs = b % kSlices;
    b /= kSlices;
    const int h = b % P.H;
    const int rank = b / P.H;

    int n, j0, nch, tok_start, L;
    if (P.cu_seqlens == nullptr) {
        n = rank;
        j0 = n * P.chunks_per_seq;
        nch = P.chunks_per_seq;
        tok_start = n * P.T;
        L = P.T;
    } else {
        if (!*M.valid) return;  // malformed cu_seqlens: write nothing
        n = M.seq_order[rank];
        j0 = M.chunk_first[n];
        nch = M.chunk_first[n + 1] - j0;
        tok_start = P.cu_seqlens[n];
        L = P.cu_seqlens[n + 1] - tok_start;
    }
    const int v0 = vs * kVS;
    const int vw = warp * 16;         // this warp's first value row inside the slice
    const size_t state_base = ((size_t)n * P.H + h) * kDim * kDim;

    // S^T accumulator fragments: Sacc[nt][i] is S[c][v] with
    //   v = v0 + vw + g + 8 (i >> 1),  c = 8 nt + 2 t + (i & 1)
    float Sacc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = v0 + vw + fg + 8 * (i >> 1);
            const int c = 8 * nt + 2 * ft + (i & 1);
            float x = 0.0f;
            if (P.init_state) {
                const size_t idx = state_base + (size_t)c * kDim + v;
                x = (P.init_dtype == KDA_F32)
                        ? static_cast<const float*>(P.init_state)[idx]
                        : __bfloat162float(static_cast<const __nv_bfloat16*>(P.init_state)[idx]);
            }
            Sacc[nt][i] = x;
        }

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nch) load_stage(S.st[s], W, (size_t)(j0 + s) * P.H + h, v0, tid);
        cp_async_commit();
    }

    const int brow_n = (lane & 7) + 8 * (lane >> 4);        // ldmatrix rows, [n][k] storage
    const int bcol_n = 8 * ((lane >> 3) & 1);
    const int brow_t = (lane & 7) + 8 * ((lane >> 3) & 1);  // ldmatrix rows, [k][n] storage
    const int bcol_t = 8 * (lane >> 4);

    for (int c = 0; c < nch; ++c) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        {
            const int cn = c + kStages - 1;
            if (cn < nch) load_stage(S.st[cn % kStages], W, (size_t)(j0 + cn) * P.H + h, v0, tid);
            cp_async_commit();
        }
        const Stage& st = S.st[c % kStages];

        // fp16 A-operand fragments of S^T (16 value rows x 128 key channels)
        uint32_t sa[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            sa[kk][0] = pack_half2(Sacc[2 * kk][0], Sacc[2 * kk][1]);
            sa[kk][1] = pack_half2(Sacc[2 * kk][2], Sacc[2 * kk][3]);
            sa[kk][2] = pack_half2(Sacc[2 * kk + 1][0], Sacc[2 * kk + 1][1]);
            sa[kk][3] = pack_half2(Sacc[2 * kk + 1][2], Sacc[2 * kk + 1][3]);
        }
        // U^T = u^T - S^T w^T  (w is stored negated), O^T = S^T qg^T
        float Uacc[2][4], Oacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 8 * nt + 2 * ft + (i & 1);
                const int v = vw + fg + 8 * (i >> 1);
                Uacc[nt][i] = __half2float(st.u[t * U_LD + v]);
                Oacc[nt][i] = 0.0f;
            }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t bw[4], bq[4];
            ldsm_x4(bw, &st.w[brow_n * LD + 16 * kk + bcol_n]);
            ldsm_x4(bq, &st.qg[brow_n * LD + 16 * kk + bcol_n]);
            mma_f16(Uacc[0], sa[kk], bw[0], bw[1]);
            mma_f16(Uacc[1], sa[kk], bw[2], bw[3]);
            mma_f16(Oacc[0], sa[kk], bq[0], bq[1]);
            mma_f16(Oacc[1], sa[kk], bq[2], bq[3]);
        }
        const uint32_t ua[4] = {pack_half2(Uacc[0][0], Uacc[0][1]),
                                pack_half2(Uacc[0][2], Uacc[0][3]),
                                pack_half2(Uacc[1][0], Uacc[1][1]),
                                pack_half2(Uacc[1][2], Uacc[1][3])};
        // O^T += U^T A_qk^T
        {
            uint32_t ba[4];
            ldsm_x4(ba, &st.aqk[brow_n * AQ_LD + bcol_n]);
            mma_f16(Oacc[0], ua, ba[0], ba[1]);
            mma_f16(Oacc[1], ua, ba[2], ba[3]);
        }
        // S^T <- S^T Diag(gc) + U^T kd
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float2 gc2 = *reinterpret_cast<const float2*>(&st.gc[8 * nt + 2 * ft]);
            Sacc[nt][0] *= gc2.x;
            Sacc[nt][1] *= gc2.y;
            Sacc[nt][2] *= gc2.x;
            Sacc[nt][3] *= gc2.y;
        }
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t bk[4];
            ldsm_x4_t(bk, &st.kd[brow_t * LD + 16 * np + bcol_t]);
            mma_f16(Sacc[2 * np], ua, bk[0], bk[1]);
            mma_f16(Sacc[2 * np + 1], ua, bk[2], bk[3]);
        }
        // outputs: stage this warp's 16 tokens x 16 value channels, then store rows
        __nv_bfloat16* os = S.ostage[warp];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 8 * nt + 2 * ft + (i & 1);
                const int v = fg + 8 * (i >> 1);
                os[t * O_LD + v] = __float2bfloat16_rn(P.scale * Oacc[nt][i]);
            }
        __syncwarp();
        {
            const int r = lane >> 1, half = lane & 1;
            const int tl = c * kChunk + r;
            if (tl < L) {
                const size_t o = ((size_t)(tok_start + tl) * P.H + h) * kDim + v0 + vw + 8 * half;
                *reinterpret_cast<uint4*>(P.out + o) =
                    *reinterpret_cast<const uint4*>(&os[r * O_LD + 8 * half]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    if (P.final_state) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = v0 + vw + fg + 8 * (i >> 1);
                const int c = 8 * nt + 2 * ft + (i & 1);
                const size_t idx = state_base + (size_t)c * kDim + v;
                if (P.final_dtype == KDA_F32)
                    static_cast<float*>(P.final_state)[idx] = Sacc[nt][i];
                else
                    static_cast<__nv_bfloat16*>(P.final_state)[idx] = __float2bfloat16_rn(Sacc[nt][i]);
            }
    }
}

bool g_attr_set[64] = {};

}  // namespace

cudaError_t launch_state(const Problem& P, const ChunkMap& M, const Workspace& W,
                         cudaStream_t s) {
    const size_t smem = sizeof(Smem);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(state_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_set[dev] = true;
    }
    const long long ctas = (long long)P.N * P.H * (kDim / kVS);
    if (ctas == 0) return cudaSuccess;
    state_kernel<<<(unsigned)ctas, kWarps * 32, smem, s>>>(P, M, W);
    return cudaGetLastError();
}

}  // namespace kda
