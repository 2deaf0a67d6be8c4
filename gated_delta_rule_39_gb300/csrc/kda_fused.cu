// Fused KDA forward kernel: one CTA per (sequence, head) runs both stages of
// the chunkwise algorithm, so q, k, v, g and beta are read from HBM once and
// only the output and the states are written.
//
//   producer warps (4)  token-parallel stage, one 16-token chunk per warp at a
//                       time, running ahead of the recurrence: gates, in-chunk
//                       cumulative base-2 log-decay G, decay-ratio products
//                       A_kk / A_qk (tf32 MMA), (I + A_kk)^-1 by forward
//                       substitution, WY factors u = T diag(b) V and
//                       w = T diag(b)(K * 2^G) (fp16 MMA), Q * 2^G,
//                       K * 2^(G_last - G), 2^G_last
//   chain warps (8)     sequential stage over the chunks: the fp32 state lives
//                       in registers as S^T fragments, 16 value rows per warp;
//                       per chunk U^T = u^T - S^T w^T, O^T = S^T (Q 2^G)^T +
//                       U^T A_qk^T, S^T <- S^T Diag(2^G_last) + U^T (K 2^(G_last-G))
//
// The stages hand chunk factors over through a 4-slot shared-memory ring
// guarded by mbarriers (full: producer -> chain, empty: chain -> producer);
// every wait is bounded and gives up with KDA_ERR_DEVICE_TIMEOUT.
//
// Chunkwise DPLR-variant (WY) algorithm with 16-token chunks, a 16 x 16
// inverse and base-2 gates: "Moonshot AI Open-Sources FlashKDA", sections
// "Why KDA?" and "What makes the kernel fast".  The pages split the two
// stages into two kernels on Hopper because the sequential stage alone left
// SMs idle; here the split stays, but inside one CTA, so the intermediate
// factors never leave shared memory.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kChainWarps = 8;              // 8 x 16 value rows = V
constexpr int kProdWarps = 4;
constexpr int kRing = 4;                    // chunk-factor slots
constexpr int kThreads = (kChainWarps + kProdWarps) * 32;
static_assert(kRing == kProdWarps, "producer p always fills slot p");

constexpr int RAW_LD = 136;   // bf16 / fp16 per padded 128-wide row (272 B)
constexpr int G_LD = 132;     // fp32 per padded row of cumulative gates
constexpr int A_LD = 17;
constexpr int TB_LD = 24;     // fp16 per row of T diag(b) (48 B)
constexpr int LD = 136;       // fp16 per padded 128-wide row of a chunk factor
constexpr int AQ_LD = 24;
constexpr int O_LD = 24;

struct ProdSmem {
    __nv_bfloat16 q[kChunk * RAW_LD];
    __nv_bfloat16 k[kChunk * RAW_LD];
    __nv_bfloat16 v[kChunk * RAW_LD];   // rewritten in place as fp16 V
    __nv_bfloat16 g[kChunk * RAW_LD];   // rewritten in place as fp16 K * 2^G
    float G[kChunk * G_LD];
    float A[kChunk * A_LD];
    __half tb[kChunk * TB_LD];
    float beta[kChunk];
};
struct Stage {
    __half qg[kChunk * LD];
    __half kd[kChunk * LD];
    __half w[kChunk * LD];     // negated
    __half u[kChunk * LD];
    __half aqk[kChunk * AQ_LD];
    float gc[kDim];
};
struct Smem {
    ProdSmem prod[kProdWarps];
    Stage st[kRing];
    __nv_bfloat16 ostage[kChainWarps][kChunk * O_LD];
    unsigned long long full[kRing];
    unsigned long long empty[kRing];
};
static_assert(sizeof(ProdSmem) % 16 == 0 && sizeof(Stage) % 16 == 0, "16-byte alignment");

// ---- mbarrier helpers ---------------------------------------------------------
__device__ __forceinline__ void mbar_init(unsigned long long* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after about 2^32 SM cycles (~2 s) and reports a timeout.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, unsigned parity, int* err) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > (1LL << 32)) {
            set_error(err, KDA_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void unpack4(uint2 raw, float (&f)[4]) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
    f[0] = __low2float(a);
    f[1] = __high2float(a);
    f[2] = __low2float(b);
    f[3] = __high2float(b);
}

struct Unit {
    int n, h, tok_start, L, nch;
};

// ---- token-parallel stage for one chunk (one warp) -------------------------------
__device__ __forceinline__ bool produce_chunk(const Problem& P, const Unit& U, int c,
                                              ProdSmem& S, Stage& st,
                                              unsigned long long* empty_bar, int lane,
                                              float expA, const float (&dtb)[4], int* err) {
    const int h = U.h;
    const int tok0 = U.tok_start + c * kChunk;
    const int len = min(kChunk, U.L - c * kChunk);
    for (int i = lane; i < kChunk * 16; i += 32) {
        const int r = i >> 4, p = i & 15;
        const int so = r * RAW_LD + p * 8;
        if (r < len) {
            const size_t go = ((size_t)(tok0 + r) * P.H + h) * kDim + p * 8;
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
        if (lane < len) b = sigmoid_fast(__bfloat162float(P.beta[(size_t)(tok0 + lane) * P.H + h]));
        S.beta[lane] = b;
    }
    const int c0 = 4 * lane;
    const float lb2 = P.lower_bound * kLog2e;
    cp_async_wait<0>();
    __syncwarp();

    // gates -> cumulative base-2 log-decay; K * 2^G later overwrites the raw g rows
    {
        float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            float gv[4];
            unpack4(*reinterpret_cast<const uint2*>(&S.g[r * RAW_LD + c0]), gv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float g2 = lb2 * sigmoid_fast(expA * (gv[i] + dtb[i]));
                run[i] += (r < len) ? g2 : 0.0f;
            }
            *reinterpret_cast<float4*>(&S.G[r * G_LD + c0]) =
                make_float4(run[0], run[1], run[2], run[3]);
        }
    }
    __syncwarp();

    // decay-ratio products A_kk, A_qk (tf32 MMA over the 128 key channels)
    const int fg = lane >> 2, ft = lane & 3;
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
        const uint32_t ak[4] = {to_tf32(k00 * e00), to_tf32(k10 * e10), to_tf32(k01 * e01),
                                to_tf32(k11 * e11)};
        const uint32_t aq[4] = {to_tf32(q00 * e00), to_tf32(q10 * e10), to_tf32(q01 * e01),
                                to_tf32(q11 * e11)};
        const uint32_t b00 = to_tf32(k00 * i00), b01 = to_tf32(k01 * i01);
        const uint32_t b10 = to_tf32(k10 * i10), b11 = to_tf32(k11 * i11);
        mma_tf32(akk[0], ak, b00, b01);
        mma_tf32(akk[1], ak, b10, b11);
        mma_tf32(aqk[0], aq, b00, b01);
        mma_tf32(aqk[1], aq, b10, b11);
    }

    // the slot must be free before anything is written into it
    const int k = c / kRing;
    if (k >= 1 && !mbar_wait(empty_bar, (unsigned)((k - 1) & 1), err)) return false;

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
            *reinterpret_cast<uint32_t*>(&st.aqk[r * AQ_LD + s]) = pack_half2(x0, x1);
        }
    __syncwarp();

    // T = (I + A_kk)^-1 by forward substitution, one column per lane; T diag(b) in fp16
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

    // fp16 operands (column-owner layout): Q 2^G, K 2^(G_last - G) into the slot;
    // K 2^G and V in place of the raw g and v rows
    __half* kg16 = reinterpret_cast<__half*>(S.g);
    __half* v16 = reinterpret_cast<__half*>(S.v);
    {
        const float4 gl4 = *reinterpret_cast<const float4*>(&S.G[(kChunk - 1) * G_LD + c0]);
        const float gl[4] = {gl4.x, gl4.y, gl4.z, gl4.w};
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
            *reinterpret_cast<uint2*>(&st.qg[r * LD + c0]) = make_uint2(
                pack_half2(qv[0] * e[0], qv[1] * e[1]), pack_half2(qv[2] * e[2], qv[3] * e[3]));
            *reinterpret_cast<uint2*>(&st.kd[r * LD + c0]) = make_uint2(
                pack_half2(kv[0] * d[0], kv[1] * d[1]), pack_half2(kv[2] * d[2], kv[3] * d[3]));
            *reinterpret_cast<uint2*>(&kg16[r * RAW_LD + c0]) = make_uint2(
                pack_half2(kv[0] * e[0], kv[1] * e[1]), pack_half2(kv[2] * e[2], kv[3] * e[3]));
            *reinterpret_cast<uint2*>(&v16[r * RAW_LD + c0]) =
                make_uint2(pack_half2(vv[0], vv[1]), pack_half2(vv[2], vv[3]));
        }
        *reinterpret_cast<float4*>(&st.gc[c0]) =
            make_float4(ex2_approx(gl[0]), ex2_approx(gl[1]), ex2_approx(gl[2]), ex2_approx(gl[3]));
    }
    __syncwarp();

    // u = T diag(b) V and w = T diag(b) (K 2^G) (stored negated), fp16 MMA, N = 128
    {
        uint32_t ta[4];
        ldsm_x4(ta, &S.tb[((lane & 7) + 8 * ((lane >> 3) & 1)) * TB_LD + 8 * (lane >> 4)]);
        const int brow = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll 2
        for (int np = 0; np < kDim / 16; ++np) {
            const int bcol = 16 * np + 8 * (lane >> 4);
            uint32_t bv[4], bk[4];
            ldsm_x4_t(bv, &v16[brow * RAW_LD + bcol]);
            ldsm_x4_t(bk, &kg16[brow * RAW_LD + bcol]);
            float cu0[4] = {}, cu1[4] = {}, cw0[4] = {}, cw1[4] = {};
            mma_f16(cu0, ta, bv[0], bv[1]);
            mma_f16(cu1, ta, bv[2], bv[3]);
            mma_f16(cw0, ta, bk[0], bk[1]);
            mma_f16(cw1, ta, bk[2], bk[3]);
            const int col0 = 16 * np + 2 * ft, col1 = col0 + 8;
            *reinterpret_cast<uint32_t*>(&st.u[fg * LD + col0]) = pack_half2(cu0[0], cu0[1]);
            *reinterpret_cast<uint32_t*>(&st.u[(fg + 8) * LD + col0]) = pack_half2(cu0[2], cu0[3]);
            *reinterpret_cast<uint32_t*>(&st.u[fg * LD + col1]) = pack_half2(cu1[0], cu1[1]);
            *reinterpret_cast<uint32_t*>(&st.u[(fg + 8) * LD + col1]) = pack_half2(cu1[2], cu1[3]);
            *reinterpret_cast<uint32_t*>(&st.w[fg * LD + col0]) = pack_half2(-cw0[0], -cw0[1]);
            *reinterpret_cast<uint32_t*>(&st.w[(fg + 8) * LD + col0]) = pack_half2(-cw0[2], -cw0[3]);
            *reinterpret_cast<uint32_t*>(&st.w[fg * LD + col1]) = pack_half2(-cw1[0], -cw1[1]);
            *reinterpret_cast<uint32_t*>(&st.w[(fg + 8) * LD + col1]) = pack_half2(-cw1[2], -cw1[3]);
        }
    }
    __syncwarp();
    return true;
}

// ---- sequential stage ------------------------------------------------------------
__device__ __forceinline__ void chain(const Problem& P, const Unit& U, Smem& S, int warp,
                                      int lane, int* err) {
    const int fg = lane >> 2, ft = lane & 3;
    const int vw = warp * 16;
    const size_t state_base = ((size_t)U.n * P.H + U.h) * kDim * kDim;

    // Sacc[nt][i] = S[c][v], v = vw + g + 8 (i >> 1), c = 8 nt + 2 t + (i & 1)
    float Sacc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = vw + fg + 8 * (i >> 1);
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

    const int brow_n = (lane & 7) + 8 * (lane >> 4);
    const int bcol_n = 8 * ((lane >> 3) & 1);
    const int brow_t = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int bcol_t = 8 * (lane >> 4);
    __nv_bfloat16* os = S.ostage[warp];

    for (int c = 0; c < U.nch; ++c) {
        const int slot = c % kRing;
        if (!mbar_wait(&S.full[slot], (unsigned)((c / kRing) & 1), err)) return;
        const Stage& st = S.st[slot];

        uint32_t sa[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            sa[kk][0] = pack_half2(Sacc[2 * kk][0], Sacc[2 * kk][1]);
            sa[kk][1] = pack_half2(Sacc[2 * kk][2], Sacc[2 * kk][3]);
            sa[kk][2] = pack_half2(Sacc[2 * kk + 1][0], Sacc[2 * kk + 1][1]);
            sa[kk][3] = pack_half2(Sacc[2 * kk + 1][2], Sacc[2 * kk + 1][3]);
        }
        float Uacc[2][4], Oacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 8 * nt + 2 * ft + (i & 1);
                const int v = vw + fg + 8 * (i >> 1);
                Uacc[nt][i] = __half2float(st.u[t * LD + v]);
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
        {
            uint32_t ba[4];
            ldsm_x4(ba, &st.aqk[brow_n * AQ_LD + bcol_n]);
            mma_f16(Oacc[0], ua, ba[0], ba[1]);
            mma_f16(Oacc[1], ua, ba[2], ba[3]);
        }
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
        // the slot's factors are all read: hand it back to its producer
        mbar_arrive(&S.empty[slot]);

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
            if (tl < U.L) {
                const size_t o = ((size_t)(U.tok_start + tl) * P.H + U.h) * kDim + vw + 8 * half;
                *reinterpret_cast<uint4*>(P.out + o) =
                    *reinterpret_cast<const uint4*>(&os[r * O_LD + 8 * half]);
            }
        }
        __syncwarp();
    }

    if (P.final_state) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = vw + fg + 8 * (i >> 1);
                const int c = 8 * nt + 2 * ft + (i & 1);
                const size_t idx = state_base + (size_t)c * kDim + v;
                if (P.final_dtype == KDA_F32)
                    static_cast<float*>(P.final_state)[idx] = Sacc[nt][i];
                else
                    static_cast<__nv_bfloat16*>(P.final_state)[idx] =
                        __float2bfloat16_rn(Sacc[nt][i]);
            }
    }
}

__global__ void __launch_bounds__(kThreads, 1) fused_kernel(Problem P, SeqMap M, int* err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    Unit U;
    U.h = blockIdx.x % P.H;
    const int rank = blockIdx.x / P.H;
    if (P.cu_seqlens == nullptr) {
        U.n = rank;
        U.tok_start = rank * P.T;
        U.L = P.T;
    } else {
        if (!*M.valid) return;  // malformed cu_seqlens: write nothing (CTA-uniform)
        U.n = M.seq_order[rank];
        U.tok_start = P.cu_seqlens[U.n];
        U.L = P.cu_seqlens[U.n + 1] - U.tok_start;
    }
    U.nch = (U.L + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&S.full[s], 32);                 // all lanes of the producer warp
            mbar_init(&S.empty[s], kChainWarps * 32);  // every chain thread
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp < kChainWarps) {
        chain(P, U, S, warp, lane, err);
    } else {
        const int pw = warp - kChainWarps;
        const float expA = expf(P.A_log[U.h]);
        const float* dtb_h = P.dt_bias + (size_t)U.h * kDim + 4 * lane;
        const float dtb[4] = {dtb_h[0], dtb_h[1], dtb_h[2], dtb_h[3]};
        for (int c = pw; c < U.nch; c += kProdWarps) {
            if (!produce_chunk(P, U, c, S.prod[pw], S.st[pw], &S.empty[pw], lane, expA, dtb, err))
                return;
            mbar_arrive(&S.full[pw]);
        }
    }
}

bool g_attr_set[64] = {};

}  // namespace

size_t fused_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_fused(const Problem& P, const SeqMap& M, int* err, cudaStream_t s) {
    const size_t smem = sizeof(Smem);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fused_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_set[dev] = true;
    }
    const long long ctas = (long long)P.N * P.H;
    if (ctas == 0) return cudaSuccess;
    fused_kernel<<<(unsigned)ctas, kThreads, smem, s>>>(P, M, err);
    return cudaGetLastError();
}

}  // namespace kda
