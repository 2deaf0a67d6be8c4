// Intra-chunk kernel: everything about one 16-token chunk of one head that
// does not depend on the recurrent state, for all chunks in parallel.
//
// For a chunk with rows r, s in 0..15 (rows past the sequence end are zero
// and carry no decay), G[r,c] = sum_{u<=r} log2-decay[u,c]:
//   A_kk[r,s] = b_r sum_c k_r[c] k_s[c] 2^(G[r,c]-G[s,c])   s <  r
//   A_qk[r,s] =     sum_c q_r[c] k_s[c] 2^(G[r,c]-G[s,c])   s <= r
//   T  = (I + A_kk)^-1 (forward substitution; A_kk is strictly lower)
//   u  = T diag(b) V          w = T diag(b) (K * 2^G)
//   qg = Q * 2^G              kd = K * 2^(G_last - G)        gc = 2^G_last
// These are the chunkwise (WY / Diagonal-Plus-Low-Rank variant) factors of
// "Moonshot AI Open-Sources FlashKDA", sections "Why KDA?" and "What makes
// the kernel fast" (chunk 16, 16x16 inverse, base-2 gates).
//
// One warp per (chunk, head); four heads of one chunk per CTA, so the four
// warps read adjacent 256-byte rows of q, k, v and g.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kWarps = 4;
constexpr int RAW_LD = 136;   // bf16 per padded 128-wide row (272 B: conflict-free, 16 B aligned)
constexpr int G_LD = 132;     // fp32 per padded row of cumulative gates
constexpr int A_LD = 17;
constexpr int TB_LD = 24;     // fp16 per row of T diag(b) (48 B rows)
constexpr int H_LD = 136;     // fp16 per padded 128-wide row

struct WarpSmem {
    __nv_bfloat16 q[kChunk * RAW_LD];
    __nv_bfloat16 k[kChunk * RAW_LD];
    __nv_bfloat16 v[kChunk * RAW_LD];
    __nv_bfloat16 g[kChunk * RAW_LD];
    float G[kChunk * G_LD];
    float A[kChunk * A_LD];
    __half tb[kChunk * TB_LD];
    __half kg16[kChunk * H_LD];
    __half v16[kChunk * H_LD];
    float beta[kChunk];
};
static_assert(sizeof(WarpSmem) % 16 == 0, "warp smem blocks must stay 16-byte aligned");

__device__ __forceinline__ void unpack4(uint2 raw, float (&f)[4]) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
    f[0] = __low2float(a);
    f[1] = __high2float(a);
    f[2] = __low2float(b);
    f[3] = __high2float(b);
}

__global__ void __launch_bounds__(kWarps * 32) intra_kernel(Problem P, ChunkMap M, Workspace W) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x;
    const int h = blockIdx.y * kWarps + warp;
    if (h >= P.H) return;  // warp-uniform; the kernel has no CTA-wide barrier
    const ChunkSpan cs = chunk_span(P, M, j);
    if (cs.seq < 0 || cs.len <= 0) return;
    WarpSmem& S = reinterpret_cast<WarpSmem*>(smem_raw)[warp];
    const size_t jh = (size_t)j * P.H + h;

    // ---- stage the chunk's rows of q, k, v, g (zero rows past the end) ------
    for (int i = lane; i < kChunk * 16; i += 32) {
        const int r = i >> 4, p = i & 15;
        const int so = r * RAW_LD + p * 8;
        if (r < cs.len) {
            const size_t go = ((size_t)(cs.tok0 + r) * P.H + h) * kDim + p * 8;
            cp_async16(&S.q[so], P.q + go);
            cp_async16(&S.k[so], P.k + go);
            cp_async16(&S.v[so], P.v + go);
            cp_async16(&S.g[so], P.g + go);
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(&S.q[so]) = z;
            *reinterpret_cast<uint4*>(&S.k[so]) = z;
            *reinterpret_cast<uint4*>(&S.v[so]) = z;
            *reinterpret_cast<uint4*>(&S.g[so]) = z;
        }
    }
    cp_async_commit();
    if (lane < kChunk) {
        float b = 0.0f;
        if (lane < cs.len)
            b = sigmoid_fast(__bfloat162float(P.beta[(size_t)(cs.tok0 + lane) * P.H + h]));
        S.beta[lane] = b;
    }
    const int c0 = 4 * lane;  // column-owner layout: this lane's 4 key channels
    const float expA = expf(P.A_log[h]);
    const float* dtb_h = P.dt_bias + (size_t)h * kDim + c0;
    const float dtb[4] = {dtb_h[0], dtb_h[1], dtb_h[2], dtb_h[3]};
    const float lb2 = P.lower_bound * kLog2e;
    cp_async_wait<0>();
    __syncwarp();

    // ---- gates: base-2 log-decay, cumulative within the chunk --------------
    {
        float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            float gv[4];
            unpack4(*reinterpret_cast<const uint2*>(&S.g[r * RAW_LD + c0]), gv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float g2 = lb2 * sigmoid_fast(expA * (gv[i] + dtb[i]));
                run[i] += (r < cs.len) ? g2 : 0.0f;
            }
            *reinterpret_cast<float4*>(&S.G[r * G_LD + c0]) =
                make_float4(run[0], run[1], run[2], run[3]);
        }
    }
    __syncwarp();

    // ---- A_kk and A_qk: tf32 MMA over the 128 key channels -----------------
    const int fg = lane >> 2, ft = lane & 3;  // fragment row group / thread-in-group
    float akk[2][4] = {}, aqk[2][4] = {};
#pragma unroll 4
    for (int kk = 0; kk < kDim / 8; ++kk) {
        const int cl = kk * 8 + ft, ch = cl + 4;
        const float G00 = S.G[fg * G_LD + cl], G01 = S.G[fg * G_LD + ch];
        const float G10 = S.G[(fg + 8) * G_LD + cl], G11 = S.G[(fg + 8) * G_LD + ch];
        const float k00 = __bfloat162float(S.k[fg * RAW_LD + cl]);
        const float k01 = __bfloat162float(S.k[fg * RAW_LD + ch]);
        const float k10 = __bfloat162float(S.k[(fg + 8) * RAW_LD + cl]);
        const float k11 = __bfloat162float(S.k[(fg + 8) * RAW_LD + ch]);
        const float q00 = __bfloat162float(S.q[fg * RAW_LD + cl]);
        const float q01 = __bfloat162float(S.q[fg * RAW_LD + ch]);
        const float q10 = __bfloat162float(S.q[(fg + 8) * RAW_LD + cl]);
        const float q11 = __bfloat162float(S.q[(fg + 8) * RAW_LD + ch]);
        const float e00 = ex2_approx(G00), e01 = ex2_approx(G01);
        const float e10 = ex2_approx(G10), e11 = ex2_approx(G11);
        const float i00 = ex2_approx(-G00), i01 = ex2_approx(-G01);
        const float i10 = ex2_approx(-G10), i11 = ex2_approx(-G11);
        // A fragment (16x8): a0 (g, t), a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4)
        const uint32_t ak[4] = {to_tf32(k00 * e00), to_tf32(k10 * e10), to_tf32(k01 * e01),
                                to_tf32(k11 * e11)};
        const uint32_t aq[4] = {to_tf32(q00 * e00), to_tf32(q10 * e10), to_tf32(q01 * e01),
                                to_tf32(q11 * e11)};
        // B fragment (8x8, B[c][s] = k_s[c] 2^-G[s,c]): b0 (c = t, s = g), b1 (c = t+4, s = g)
        const uint32_t b00 = to_tf32(k00 * i00), b01 = to_tf32(k01 * i01);
        const uint32_t b10 = to_tf32(k10 * i10), b11 = to_tf32(k11 * i11);
        mma_tf32(akk[0], ak, b00, b01);
        mma_tf32(akk[1], ak, b10, b11);
        mma_tf32(aqk[0], aq, b00, b01);
        mma_tf32(aqk[1], aq, b10, b11);
    }
    // accumulator element i of n-tile nt: row r = g + 8(i>>1), column s = 8 nt + 2t + (i&1)
    {
        __half* aq_out = W.aqk + jh * (kChunk * kChunk);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
                const int r = fg + 8 * hi;
                const int s = 8 * nt + 2 * ft;
                const float br = S.beta[r];
                S.A[r * A_LD + s] = (s < r) ? br * akk[nt][2 * hi] : 0.0f;
                S.A[r * A_LD + s + 1] = (s + 1 < r) ? br * akk[nt][2 * hi + 1] : 0.0f;
                const float x0 = (s <= r) ? aqk[nt][2 * hi] : 0.0f;
                const float x1 = (s + 1 <= r) ? aqk[nt][2 * hi + 1] : 0.0f;
                *reinterpret_cast<uint32_t*>(&aq_out[r * kChunk + s]) = pack_half2(x0, x1);
            }
    }
    __syncwarp();

    // ---- T = (I + A_kk)^-1 by forward substitution, one column per lane ----
    if (lane < kChunk) {
        float Tc[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            float s = 0.0f;
#pragma unroll
            for (int m = 0; m < i; ++m) s = fmaf(S.A[i * A_LD + m], Tc[m], s);
            Tc[i] = (i == lane) ? 1.0f : ((i < lane) ? 0.0f : -s);
        }
        const float bj = S.beta[lane];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) S.tb[i * TB_LD + lane] = __float2half_rn(Tc[i] * bj);
    }

    // ---- fp16 operands for the state recurrence (column-owner layout) ------
    {
        const float4 gl4 = *reinterpret_cast<const float4*>(&S.G[(kChunk - 1) * G_LD + c0]);
        const float gl[4] = {gl4.x, gl4.y, gl4.z, gl4.w};
        __half* qg_out = W.qg + jh * (kChunk * kDim);
        __half* kd_out = W.kd + jh * (kChunk * kDim);
#pragma unroll 4
        for (int r = 0; r < kChunk; ++r) {
            const float4 G4 = *reinterpret_cast<const float4*>(&S.G[r * G_LD + c0]);
            const float Gr[4] = {G4.x, G4.y, G4.z, G4.w};
            float kv[4], qv[4], vv[4];
            unpack4(*reinterpret_cast<const uint2*>(&S.k[r * RAW_LD + c0]), kv);
            unpack4(*reinterpret_cast<const uint2*>(&S.q[r * RAW_LD + c0]), qv);
            unpack4(*reinterpret_cast<const uint2*>(&S.v[r * RAW_LD + c0]), vv);
            float e[4], d[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                e[i] = ex2_approx(Gr[i]);
                d[i] = ex2_approx(gl[i] - Gr[i]);
            }
            const uint2 qg2 = make_uint2(pack_half2(qv[0] * e[0], qv[1] * e[1]),
                                         pack_half2(qv[2] * e[2], qv[3] * e[3]));
            const uint2 kd2 = make_uint2(pack_half2(kv[0] * d[0], kv[1] * d[1]),
                                         pack_half2(kv[2] * d[2], kv[3] * d[3]));
            const uint2 kg2 = make_uint2(pack_half2(kv[0] * e[0], kv[1] * e[1]),
                                         pack_half2(kv[2] * e[2], kv[3] * e[3]));
            const uint2 v2 = make_uint2(pack_half2(vv[0], vv[1]), pack_half2(vv[2], vv[3]));
            *reinterpret_cast<uint2*>(&qg_out[r * kDim + c0]) = qg2;
            *reinterpret_cast<uint2*>(&kd_out[r * kDim + c0]) = kd2;
            *reinterpret_cast<uint2*>(&S.kg16[r * H_LD + c0]) = kg2;
            *reinterpret_cast<uint2*>(&S.v16[r * H_LD + c0]) = v2;
        }
        float e4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) e4[i] = ex2_approx(gl[i]);
        *reinterpret_cast<float4*>(W.gc + jh * kDim + c0) = make_float4(e4[0], e4[1], e4[2], e4[3]);
    }
    __syncwarp();

    // ---- u = T diag(b) V and w = T diag(b) (K * 2^G): fp16 MMA, N = 128 ------
    __half* ust = reinterpret_cast<__half*>(S.q);  // staging (q, k rows no longer needed)
    __half* wst = reinterpret_cast<__half*>(S.k);
    {
        uint32_t ta[4];
        ldsm_x4(ta, &S.tb[((lane & 7) + 8 * ((lane >> 3) & 1)) * TB_LD + 8 * (lane >> 4)]);
#pragma unroll 2
        for (int np = 0; np < kDim / 16; ++np) {
            const int brow = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int bcol = 16 * np + 8 * (lane >> 4);
            uint32_t bv[4], bk[4];
            ldsm_x4_t(bv, &S.v16[brow * H_LD + bcol]);
            ldsm_x4_t(bk, &S.kg16[brow * H_LD + bcol]);
            float cu0[4] = {}, cu1[4] = {}, cw0[4] = {}, cw1[4] = {};
            mma_f16(cu0, ta, bv[0], bv[1]);
            mma_f16(cu1, ta, bv[2], bv[3]);
            mma_f16(cw0, ta, bk[0], bk[1]);
            mma_f16(cw1, ta, bk[2], bk[3]);
            const int col0 = 16 * np + 2 * ft, col1 = col0 + 8;
            *reinterpret_cast<uint32_t*>(&ust[fg * H_LD + col0]) = pack_half2(cu0[0], cu0[1]);
            *reinterpret_cast<uint32_t*>(&ust[(fg + 8) * H_LD + col0]) = pack_half2(cu0[2], cu0[3]);
            *reinterpret_cast<uint32_t*>(&ust[fg * H_LD + col1]) = pack_half2(cu1[0], cu1[1]);
            *reinterpret_cast<uint32_t*>(&ust[(fg + 8) * H_LD + col1]) = pack_half2(cu1[2], cu1[3]);
            *reinterpret_cast<uint32_t*>(&wst[fg * H_LD + col0]) = pack_half2(-cw0[0], -cw0[1]);
            *reinterpret_cast<uint32_t*>(&wst[(fg + 8) * H_LD + col0]) = pack_half2(-cw0[2], -cw0[3]);
            *reinterpret_cast<uint32_t*>(&wst[fg * H_LD + col1]) = pack_half2(-cw1[0], -cw1[1]);
            *reinterpret_cast<uint32_t*>(&wst[(fg + 8) * H_LD + col1]) = pack_half2(-cw1[2], -cw1[3]);
        }
    }
    __syncwarp();
    {
        __half* u_out = W.u + jh * (kChunk * kDim);
        __half* w_out = W.wneg + jh * (kChunk * kDim);
        for (int i = lane; i < kChunk * 16; i += 32) {
            const int r = i >> 4, p = i & 15;
            *reinterpret_cast<uint4*>(&u_out[r * kDim + p * 8]) =
                *reinterpret_cast<const uint4*>(&ust[r * H_LD + p * 8]);
            *reinterpret_cast<uint4*>(&w_out[r * kDim + p * 8]) =
                *reinterpret_cast<const uint4*>(&wst[r * H_LD + p * 8]);
        }
    }
}

bool g_attr_set[64] = {};

}  // namespace

cudaError_t launch_intra(const Problem& P, const ChunkMap& M, const Workspace& W,
                         cudaStream_t s) {
    const size_t smem = sizeof(WarpSmem) * kWarps;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(intra_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_set[dev] = true;
    }
    dim3 grid(P.chunk_bound, (P.H + kWarps - 1) / kWarps);
    intra_kernel<<<grid, kWarps * 32, smem, s>>>(P, M, W);
    return cudaGetLastError();
}

}  // namespace kda
