// Fused KDA forward kernel: one CTA per (sequence, head) runs both stages of
// the chunkwise algorithm, so q, k, v, g and beta are read from HBM once and
// only the output and the states are written.
//
//   producer warps (8)  the token-parallel stage.  Warp w owns key / value
//                       channels 16w .. 16w+15 of every 16-token chunk: it loads
//                       its slice of q, k, v, g straight into registers (one chunk
//                       ahead), computes the gates and their in-chunk cumulative
//                       sum across rows with warp shuffles, the decay factors,
//                       the operand tiles of the recurrence (Q 2^G, K 2^(G_last-G),
//                       V, 2^G_last) and its share of the decay-ratio products
//                       A_kk and A_qk (tf32 MMA fed from registers, summed across
//                       warps in shared memory).  One chunk later it forms its
//                       slice of w = T diag(b)(K 2^G).
//   solver warp         (I + A_kk)^-1 by forward substitution, T diag(b), A_qk.
//   MMA warp            issues the tcgen05 MMAs of the recurrence (one thread).
//   epilogue warps (4)  own the tensor-memory state S^T (lane v = value channel v).
//
// Chunkwise DPLR-variant (WY) algorithm with 16-token chunks, a 16 x 16
// inverse and base-2 gates: "Moonshot AI Open-Sources FlashKDA", sections
// "Why KDA?" and "What makes the kernel fast".  The pages split the two
// stages into two kernels on Hopper because the sequential stage alone left
// SMs idle; here the split stays, but inside one CTA, so the intermediate
// factors never leave the SM.
#include "kda_internal.cuh"
#include "kda_tcgen05.cuh"

namespace kda {

namespace {

constexpr int kEpiWarps = 8;                // epilogue: two warps per TMEM lane quarter,
                                            // each owning half of the state's columns
constexpr int kMmaWarp = kEpiWarps;         // issues the tcgen05 MMAs, owns tensor memory
constexpr int kSolveWarp = kMmaWarp + 1;    // 16 x 16 inverse
constexpr int kProdWarp0 = kSolveWarp + 1;
constexpr int kProdWarps = 8;               // 16 key channels each
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kRing = 6;                    // chunk-operand slots
constexpr int kThreads = (kProdWarp0 + kProdWarps) * 32;

constexpr int A_LD = 17;
constexpr int TB_LD = 24;     // fp16 per row of T diag(b) (48 B: ldmatrix conflict-free)
constexpr int KG_LD = 24;     // fp16 per row of a warp's K 2^G tile (48 B)
constexpr int T_SBO = 272;    // byte step between 8-row groups of the transposed 128 x 16
                              // tiles (16 bytes past 256 spreads row groups over banks)

// tensor-memory columns (one allocation of 512)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S32 = 0;     // S^T, fp32, 128 columns
constexpr uint32_t TM_S16 = 128;   // S^T as the fp16 A operand, 64 columns
constexpr uint32_t TM_UO = 192;    // [U | O] accumulators, 2 buffers x 32 columns
constexpr uint32_t TM_U16 = 256;   // U^T as the fp16 A operand, 8 columns

// One chunk's operands for the tensor-core recurrence (canonical K-major layouts)
struct Stage {
    __half buo[2 * 32 * 64];       // B of [U|O] += S^T [-w; Q 2^G]^T: 32 x 128, 128B swizzle
    __half vt[16 * T_SBO / 2];     // A of u^T = V^T (T diag b)^T: V^T 128 x 16, interleaved
    __half kdt[16 * T_SBO / 2];    // B of the state update: (K 2^(G_last-G))^T 128 x 16
    __half tbt[32 * 16];           // B of the u MMA: rows 0-15 T diag(b), rows 16-31 zero
    __half aqk[16 * 16];           // B of O += U A_qk^T: A_qk 16 x 16
    float gc[kDim];                // 2^G_last
    unsigned char pad_[512];       // keep sizeof(Stage) a multiple of 1024
};
static_assert(sizeof(Stage) % 1024 == 0, "stages keep the swizzled tiles 1024-byte aligned");
struct ProdShared {
    float part[2][kProdWarps][2][kChunk * kChunk]; // [chunk parity][warp][A_kk, A_qk] partials
    __half tb[2][kChunk * TB_LD];                  // T diag(b) per chunk parity
    __half kg[kProdWarps][2][kChunk * KG_LD];      // each warp's K 2^G tile per chunk parity
    float A[kChunk * A_LD];                        // solver scratch
};
struct Smem {
    Stage st[kRing];
    ProdShared pr;
    unsigned long long full[kRing];    // producers -> MMA / epilogue
    unsigned long long empty[kRing];   // MMA commit -> producers
    unsigned long long a_ready[2];     // producers' partial A_kk / A_qk summed
    unsigned long long t_ready[2];     // solver: T diag(b), A_qk written
    unsigned long long uo_done;        // U|O MMAs complete
    unsigned long long s_done;         // state update + O MMAs complete
    unsigned long long s16_ready;      // epilogue: S^T fp16 copy written, S^T rescaled
    unsigned long long u16_ready;      // epilogue: U^T fp16 copy written
    unsigned long long epi_done;       // epilogue finished with tensor memory
    uint32_t tmem_base;
};

// ---- small helpers ------------------------------------------------------------
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
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(1000000u)   // may sleep up to 1 ms per try
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
// packed fp32 pair arithmetic (one instruction each on sm_100 and later)
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) {
    unsigned long long x, y, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("mul.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(z));
    return r;
}
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) {
    unsigned long long x, y, w, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(w) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(z) : "l"(x), "l"(y), "l"(w));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(z));
    return r;
}
// packed fp32 pair multiply (one instruction on sm_100 and later)
__device__ __forceinline__ void mul2(float& a, float& b, float2 s) {
    unsigned long long x, y, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(s.x), "f"(s.y));
    asm("mul.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(z));
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t raw) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&raw);
    return __bfloat1622float2(v);
}
__device__ __forceinline__ float tf32_round(float x) { return __uint_as_float(to_tf32(x)); }

struct Unit {
    int n, h, tok_start, L, nch;
};

// ---- token-parallel stage: producer warp w, channels 16w .. 16w+15 ----------------
// Lane (g, t) = (lane >> 2, lane & 3) holds rows g and g+8 of the chunk for the
// channel pairs p = 16w + 8kk + 2t, p+1 (kk = 0, 1).  In the tf32 MMA fragments
// of k-step kk the pair plays logical columns t and t+4; the decay-ratio
// products sum over channels, so this relabelling leaves them unchanged.
struct RawSlice {
    uint32_t q[2][2], k[2][2], v[2][2], g[2][2];   // [row g / g+8][kk] bf16 pairs
};

__device__ __forceinline__ void load_slice(const Problem& P, const Unit& U, int c, int cbase,
                                           int lg, int lt, RawSlice& X) {
    const int len = min(kChunk, U.L - c * kChunk);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = lg + 8 * i;
        const bool ok = r < len;
        const size_t row = ((size_t)(U.tok_start + c * kChunk + (ok ? r : 0)) * P.H + U.h) * kDim;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const size_t o = row + cbase + 8 * kk + 2 * lt;
            X.q[i][kk] = ok ? __ldg(reinterpret_cast<const unsigned int*>(P.q + o)) : 0u;
            X.k[i][kk] = ok ? __ldg(reinterpret_cast<const unsigned int*>(P.k + o)) : 0u;
            X.v[i][kk] = ok ? __ldg(reinterpret_cast<const unsigned int*>(P.v + o)) : 0u;
            X.g[i][kk] = ok ? __ldg(reinterpret_cast<const unsigned int*>(P.g + o)) : 0u;
        }
    }
}

__device__ void produce(const Problem& P, const Unit& U, Smem& S, int w, int lane, int* err) {
    const int lg = lane >> 2, lt = lane & 3;
    const int cbase = 16 * w;
    const float expA = expf(P.A_log[U.h]);
    const float ga = -expA * kLog2e;   // sigmoid argument in base 2: g ga + gb
    float gb[2][2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int e = 0; e < 2; ++e) gb[kk][e] = ga * P.dt_bias[(size_t)U.h * kDim + cbase + 8 * kk + 2 * lt + e];
    const float lb2 = P.lower_bound * kLog2e;
    ProdShared& PS = S.pr;

    RawSlice nxt;
    if (U.nch > 0) load_slice(P, U, 0, cbase, lg, lt, nxt);

    for (int c = 0; c <= U.nch; ++c) {
        if (c < U.nch) {
            const RawSlice X = nxt;
            if (c + 1 < U.nch) load_slice(P, U, c + 1, cbase, lg, lt, nxt);
            const int len = min(kChunk, U.L - c * kChunk);
            const int slot = c % kRing;
            Stage& st = S.st[slot];
            const int par = c & 1;
            bool ok = true;
            if (c >= kRing) ok = mbar_wait(&S.empty[slot], (unsigned)(((c / kRing) - 1) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return;

            // gates, cumulative over rows: Hillis-Steele scan across the 8 lanes of equal t
            float G[2][2][2];   // [row g / g+8][kk][e]
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const float2 gv = bf2_to_f2(X.g[i][kk]);
                    const bool valid = lg + 8 * i < len;
                    const float2 xa = f2fma(gv, make_float2(ga, ga), make_float2(gb[kk][0], gb[kk][1]));
                    const float2 sg = f2mul(make_float2(rcp_approx(1.0f + ex2_approx(xa.x)),
                                                        rcp_approx(1.0f + ex2_approx(xa.y))),
                                            make_float2(lb2, lb2));
                    G[i][kk][0] = valid ? sg.x : 0.0f;
                    G[i][kk][1] = valid ? sg.y : 0.0f;
                }
            float glast[2][2];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float a = G[0][kk][e], b = G[1][kk][e];
#pragma unroll
                    for (int d = 4; d < 32; d <<= 1) {
                        const float ya = __shfl_up_sync(0xffffffffu, a, d);
                        const float yb = __shfl_up_sync(0xffffffffu, b, d);
                        if (lane >= d) {
                            a += ya;
                            b += yb;
                        }
                    }
                    const float tot = __shfl_sync(0xffffffffu, a, 28 + lt);   // rows 0..7
                    G[0][kk][e] = a;
                    G[1][kk][e] = tot + b;
                    glast[kk][e] = __shfl_sync(0xffffffffu, tot + b, 28 + lt);   // row 15
                }

            // decay factors and operand tiles
            unsigned char* buo = reinterpret_cast<unsigned char*>(st.buo);
            unsigned char* kdt = reinterpret_cast<unsigned char*>(st.kdt);
            unsigned char* vt = reinterpret_cast<unsigned char*>(st.vt);
            __half* kgt = PS.kg[w][par];
            uint32_t akf[2][4], aqf[2][4], bf0[2][2], bf1[2][2];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int p = cbase + 8 * kk + 2 * lt;
                const float gc0 = ex2_approx(glast[kk][0]), gc1 = ex2_approx(glast[kk][1]);
                if (lg == 0) *reinterpret_cast<float2*>(&st.gc[p]) = make_float2(gc0, gc1);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = lg + 8 * i;
                    const float e0 = ex2_approx(G[i][kk][0]), e1 = ex2_approx(G[i][kk][1]);
                    const float d0 = ex2_approx(-G[i][kk][0]), d1 = ex2_approx(-G[i][kk][1]);
                    const float2 kv = bf2_to_f2(X.k[i][kk]);
                    const float2 qv = bf2_to_f2(X.q[i][kk]);
                    const float2 vv = bf2_to_f2(X.v[i][kk]);
                    const float2 kg = f2mul(kv, make_float2(e0, e1));
                    const float2 ki = f2mul(kv, make_float2(d0, d1));
                    const float2 qg = f2mul(qv, make_float2(e0, e1));
                    const float2 kd = f2mul(ki, make_float2(gc0, gc1));
                    const float kg0 = kg.x, kg1 = kg.y, ki0 = ki.x, ki1 = ki.y, qg0 = qg.x, qg1 = qg.y;
                    // tf32 fragments: A rows g / g+8 -> a0,a2 / a1,a3; B n-tile i
                    akf[kk][i] = to_tf32(kg0);
                    akf[kk][i + 2] = to_tf32(kg1);
                    aqf[kk][i] = to_tf32(qg0);
                    aqf[kk][i + 2] = to_tf32(qg1);
                    if (i == 0) {
                        bf0[kk][0] = to_tf32(ki0);
                        bf0[kk][1] = to_tf32(ki1);
                    } else {
                        bf1[kk][0] = to_tf32(ki0);
                        bf1[kk][1] = to_tf32(ki1);
                    }
                    *reinterpret_cast<uint32_t*>(buo + tc::swizzled_offset(16 + r, p, 32)) =
                        pack_half2(qg0, qg1);
                    *reinterpret_cast<uint32_t*>(&kgt[r * KG_LD + 8 * kk + 2 * lt]) =
                        pack_half2(kg0, kg1);
                    *reinterpret_cast<__half*>(kdt + tc::interleaved16_offset(p, r, T_SBO)) =
                        __float2half_rn(kd.x);
                    *reinterpret_cast<__half*>(kdt + tc::interleaved16_offset(p + 1, r, T_SBO)) =
                        __float2half_rn(kd.y);
                    *reinterpret_cast<__half*>(vt + tc::interleaved16_offset(p, r, T_SBO)) =
                        __float2half_rn(vv.x);
                    *reinterpret_cast<__half*>(vt + tc::interleaved16_offset(p + 1, r, T_SBO)) =
                        __float2half_rn(vv.y);
                }
            }
            // this warp's share of A_kk = (K 2^G)(K 2^-G)^T and A_qk = (Q 2^G)(K 2^-G)^T
            float pk[2][4] = {}, pq[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                mma_tf32(pk[0], akf[kk], bf0[kk][0], bf0[kk][1]);
                mma_tf32(pk[1], akf[kk], bf1[kk][0], bf1[kk][1]);
                mma_tf32(pq[0], aqf[kk], bf0[kk][0], bf0[kk][1]);
                mma_tf32(pq[1], aqf[kk], bf1[kk][0], bf1[kk][1]);
            }
            // partials go to this warp's own slots; the solver sums them in a fixed
            // order, so results do not depend on warp timing
            float* ak = PS.part[par][w][0];
            float* aq = PS.part[par][w][1];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int e = (lg + 8 * hh) * kChunk + 8 * nt + 2 * lt;
                    *reinterpret_cast<float2*>(&ak[e]) = make_float2(pk[nt][2 * hh], pk[nt][2 * hh + 1]);
                    *reinterpret_cast<float2*>(&aq[e]) = make_float2(pq[nt][2 * hh], pq[nt][2 * hh + 1]);
                }
            mbar_arrive(&S.a_ready[par]);
        }
        // ---- one chunk behind: w = T diag(b)(K 2^G) for this warp's channels -------
        if (c >= 1) {
            const int cp = c - 1;
            const int par = cp & 1;
            const bool ok = mbar_wait(&S.t_ready[par], (unsigned)((cp >> 1) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return;
            Stage& st = S.st[cp % kRing];
            unsigned char* buo = reinterpret_cast<unsigned char*>(st.buo);
            uint32_t ta[4], b[4];
            ldsm_x4(ta, &PS.tb[par][((lane & 7) + 8 * ((lane >> 3) & 1)) * TB_LD + 8 * (lane >> 4)]);
            ldsm_x4_t(b, &PS.kg[w][par][((lane & 7) + 8 * ((lane >> 3) & 1)) * KG_LD + 8 * (lane >> 4)]);
            float cw0[4] = {}, cw1[4] = {};
            mma_f16(cw0, ta, b[0], b[1]);
            mma_f16(cw1, ta, b[2], b[3]);
            const int col0 = cbase + 2 * lt, col1 = col0 + 8;
            *reinterpret_cast<uint32_t*>(buo + tc::swizzled_offset(lg, col0, 32)) = pack_half2(-cw0[0], -cw0[1]);
            *reinterpret_cast<uint32_t*>(buo + tc::swizzled_offset(lg + 8, col0, 32)) = pack_half2(-cw0[2], -cw0[3]);
            *reinterpret_cast<uint32_t*>(buo + tc::swizzled_offset(lg, col1, 32)) = pack_half2(-cw1[0], -cw1[1]);
            *reinterpret_cast<uint32_t*>(buo + tc::swizzled_offset(lg + 8, col1, 32)) = pack_half2(-cw1[2], -cw1[3]);
            // generic-proxy writes of this thread -> visible to the tensor core
            tc::fence_proxy_async_smem();
            mbar_arrive(&S.full[cp % kRing]);
        }
    }
}

// ---- solver warp: (I + A_kk)^-1, T diag(b), A_qk for every chunk ------------------
__device__ void solve(const Problem& P, const Unit& U, Smem& S, int lane, int* err) {
    ProdShared& PS = S.pr;
    const size_t beta_base = (size_t)U.tok_start * P.H + U.h;
    float logit = 0.0f;
    if (U.nch > 0 && lane < kChunk && lane < U.L)
        logit = __bfloat162float(P.beta[beta_base + (size_t)lane * P.H]);
    for (int c = 0; c < U.nch; ++c) {
        const int len = min(kChunk, U.L - c * kChunk);
        const float bl = (lane < len) ? sigmoid_fast(logit) : 0.0f;   // b of row `lane`
        if (c + 1 < U.nch && lane < kChunk && (c + 1) * kChunk + lane < U.L)
            logit = __bfloat162float(P.beta[beta_base + (size_t)((c + 1) * kChunk + lane) * P.H]);
        const int par = c & 1;
        const bool ok = mbar_wait(&S.a_ready[par], (unsigned)((c >> 1) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return;
        Stage& st = S.st[c % kRing];
        // A_kk = diag(b) (sum of the warps' partials), strictly lower; A_qk inclusive
        // lower (fp16, interleaved); partials summed in warp order
#pragma unroll
        for (int e = 2 * lane; e < kChunk * kChunk; e += 64) {
            const int r = e >> 4, s = e & 15;
            float2 sk = make_float2(0.f, 0.f), sq = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kProdWarps; ++w) {
                const float2 pk2 = *reinterpret_cast<const float2*>(&PS.part[par][w][0][e]);
                const float2 pq2 = *reinterpret_cast<const float2*>(&PS.part[par][w][1][e]);
                sk.x += pk2.x;
                sk.y += pk2.y;
                sq.x += pq2.x;
                sq.y += pq2.y;
            }
            const float br = __shfl_sync(0xffffffffu, bl, r);
            PS.A[r * A_LD + s] = (s < r) ? br * sk.x : 0.0f;
            PS.A[r * A_LD + s + 1] = (s + 1 < r) ? br * sk.y : 0.0f;
            *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(st.aqk) +
                                         tc::interleaved_offset(r, s, kChunk)) =
                pack_half2((s <= r) ? sq.x : 0.0f, (s + 1 <= r) ? sq.y : 0.0f);
        }
        __syncwarp();
        if (lane < kChunk) {
            float Tc[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                for (int m = 0; m + 1 < i; m += 2) {
                    s0 = fmaf(PS.A[i * A_LD + m], Tc[m], s0);
                    s1 = fmaf(PS.A[i * A_LD + m + 1], Tc[m + 1], s1);
                }
                if (i & 1) s0 = fmaf(PS.A[i * A_LD + i - 1], Tc[i - 1], s0);
                Tc[i] = (i == lane) ? 1.0f : ((i < lane) ? 0.0f : -(s0 + s1));
            }
            unsigned char* tbt = reinterpret_cast<unsigned char*>(st.tbt);
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const __half x = __float2half_rn(Tc[i] * bl);
                PS.tb[par][i * TB_LD + lane] = x;
                *reinterpret_cast<__half*>(tbt + tc::interleaved_offset(i, lane, kChunk)) = x;
            }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive(&S.t_ready[par]);
    }
}

// ---- sequential stage: tensor-core issue (one thread) -------------------------------
// Per chunk c (slot s), in the transposed orientation (TMEM lane = value row v):
//   [U|O] = V^T [T diag(b) ; 0]^T             (u^T into the U half, zeros into O)
//   [U|O] += S^T [-w ; Q 2^G]^T               (8 MMAs over the 128 key channels)
//   S^T  += U^T (K 2^(G_last-G))              (S^T was rescaled by 2^G_last beforehand)
//   O    += U^T A_qk^T
__device__ void mma_issuer(const Unit& U, Smem& S, uint32_t tmem, int* err) {
    constexpr uint32_t id32 = tc::idesc_f16_f32(128, 32);
    constexpr uint32_t id16 = tc::idesc_f16_f32(128, 16);
    constexpr uint32_t id128 = tc::idesc_f16_f32(128, 128);
    for (int c = 0; c < U.nch; ++c) {
        const int slot = c % kRing;
        const Stage& st = S.st[slot];
        const uint32_t uo = tmem + TM_UO + 32u * (c & 1);
        if (!mbar_wait(&S.full[slot], (unsigned)((c / kRing) & 1), err)) return;
        if (!mbar_wait(&S.s16_ready, (unsigned)(c & 1), err)) return;
        tc::fence_after_sync();
        tc::mma_ss(uo, tc::smem_desc(smem_u32(st.vt), 128, T_SBO, tc::kSwizzleNone),
                   tc::smem_desc(smem_u32(st.tbt), 128, 256, tc::kSwizzleNone), id32, 0);
        const uint32_t buo = smem_u32(st.buo);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t b = buo + (kk >> 2) * (32 * 128) + (kk & 3) * 32;
            tc::mma_ts(uo, tmem + TM_S16 + 8 * kk, tc::smem_desc(b, 16, 1024, tc::kSwizzle128B),
                       id32, 1);
        }
        tc::commit(smem_u32(&S.uo_done));
        if (!mbar_wait(&S.u16_ready, (unsigned)(c & 1), err)) return;
        tc::fence_after_sync();
        tc::mma_ts(tmem + TM_S32, tmem + TM_U16,
                   tc::smem_desc(smem_u32(st.kdt), 128, T_SBO, tc::kSwizzleNone), id128, 1);
        tc::mma_ts(uo + 16, tmem + TM_U16,
                   tc::smem_desc(smem_u32(st.aqk), 128, 256, tc::kSwizzleNone), id16, 1);
        tc::commit(smem_u32(&S.s_done));
        tc::commit(smem_u32(&S.empty[slot]));
    }
}

__device__ __forceinline__ float state_in(const Problem& P, size_t idx) {
    return (P.init_dtype == KDA_F32)
               ? static_cast<const float*>(P.init_state)[idx]
               : __bfloat162float(static_cast<const __nv_bfloat16*>(P.init_state)[idx]);
}
__device__ __forceinline__ void state_out(const Problem& P, size_t idx, float x) {
    if (P.final_dtype == KDA_F32)
        static_cast<float*>(P.final_state)[idx] = x;
    else
        static_cast<__nv_bfloat16*>(P.final_state)[idx] = __float2bfloat16_rn(x);
}

// ---- sequential stage: epilogue ---------------------------------------------------
// Warp ew reaches TMEM lanes 32 (ew % 4) .. + 31 (thread = value channel v) and
// owns half of the state's columns: key channels 64 (ew / 4) .. + 63, U columns
// (tokens) 8 (ew / 4) .. + 7 and the outputs of those tokens.  After each state
// update it first writes the fp16 copy that the next chunk's MMAs read (the
// critical path), then pre-scales the fp32 state by the next chunk's 2^G_last.
__device__ __forceinline__ void scale32(uint32_t (&x)[32], const float* gc) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gc + i);
        const float2 a = f2mul(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])),
                               make_float2(g4.x, g4.y));
        const float2 b = f2mul(make_float2(__uint_as_float(x[i + 2]), __uint_as_float(x[i + 3])),
                               make_float2(g4.z, g4.w));
        x[i] = __float_as_uint(a.x);
        x[i + 1] = __float_as_uint(a.y);
        x[i + 2] = __float_as_uint(b.x);
        x[i + 3] = __float_as_uint(b.y);
    }
}
__device__ __forceinline__ void pack32(const uint32_t (&x)[32], uint32_t (&h)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        h[i] = pack_half2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
}

__device__ void epilogue(const Problem& P, const Unit& U, Smem& S, uint32_t tmem, int ew,
                         int lane, int* err) {
    const int quarter = ew & 3, colhalf = ew >> 2;
    const int v = 32 * quarter + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);   // this warp's lane quarter
    const size_t sbase = ((size_t)U.n * P.H + U.h) * kDim * kDim + v;   // + c * kDim
    const int p0 = 2 * colhalf;   // this warp's two 32-column pieces: p0, p0 + 1
    bool ok = true;

    if (U.nch == 0) {   // no tokens: the final state is the initial state
        if (P.final_state)
            for (int c = 64 * colhalf; c < 64 * colhalf + 64; ++c)
                state_out(P, sbase + (size_t)c * kDim,
                          P.init_state ? state_in(P, sbase + (size_t)c * kDim) : 0.0f);
        return;
    }
    // initial state: S16 = fp16(S0), S32 = S0 Diag(2^G_last of chunk 0)
    ok = mbar_wait(&S.full[0], 0u, err);
    if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll 1
    for (int piece = p0; piece < p0 + 2; ++piece) {
        uint32_t x[32], h[16];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = 32 * piece + i;
            x[i] = __float_as_uint(P.init_state ? state_in(P, sbase + (size_t)c * kDim) : 0.0f);
        }
        pack32(x, h);
        tc::st16(tl + TM_S16 + 16 * piece, h);
        scale32(x, S.st[0].gc + 32 * piece);
        tc::st32(tl + TM_S32 + 32 * piece, x);
    }
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(&S.s16_ready);

    for (int c = 0; c < U.nch; ++c) {
        const uint32_t uo = tl + TM_UO + 32u * (c & 1);
        // U^T (this warp's 8 token columns) -> fp16 A operand of the update
        ok = mbar_wait(&S.uo_done, (unsigned)(c & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc::fence_after_sync();
        {
            uint32_t u[16], h[8];
            tc::ld16(uo, u);   // all 16 columns (one instruction); this warp converts its half
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                h[i] = pack_half2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
            if (colhalf == 0) tc::st8(tl + TM_U16, h);
            tc::wait_st();
        }
        tc::fence_before_sync();
        mbar_arrive(&S.u16_ready);

        // state update done: fp16 copy first (next chunk's MMAs wait on it) ...
        ok = mbar_wait(&S.s_done, (unsigned)(c & 1), err);
        const bool more = c + 1 < U.nch;
        const int nslot = (c + 1) % kRing;
        if (more) ok = ok && mbar_wait(&S.full[nslot], (unsigned)(((c + 1) / kRing) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc::fence_after_sync();
        if (more) {
#pragma unroll 1
            for (int piece = p0; piece < p0 + 2; ++piece) {
                uint32_t x[32], h[16];
                tc::ld32(tl + TM_S32 + 32 * piece, x);
                tc::wait_ld();
                pack32(x, h);
                tc::st16(tl + TM_S16 + 16 * piece, h);
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(&S.s16_ready);
            // ... then the rescale, finished before this warp's next U^T arrive (which
            // the next state update waits for)
#pragma unroll 1
            for (int piece = p0; piece < p0 + 2; ++piece) {
                uint32_t x[32];
                tc::ld32(tl + TM_S32 + 32 * piece, x);
                tc::wait_ld();
                scale32(x, S.st[nslot].gc + 32 * piece);
                tc::st32(tl + TM_S32 + 32 * piece, x);
            }
        } else if (P.final_state) {
#pragma unroll 1
            for (int piece = p0; piece < p0 + 2; ++piece) {
                uint32_t x[32];
                tc::ld32(tl + TM_S32 + 32 * piece, x);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    state_out(P, sbase + (size_t)(32 * piece + i) * kDim, __uint_as_float(x[i]));
            }
        }
        // outputs of chunk c, tokens 8 colhalf .. + 7: O^T lane v, column t
        {
            uint32_t o[16];
            tc::ld16(uo + 16, o);
            tc::wait_ld();
            const int len = min(kChunk, U.L - c * kChunk);
            __nv_bfloat16* out = P.out + ((size_t)(U.tok_start + c * kChunk) * P.H + U.h) * kDim + v;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = 8 * colhalf + j;
                const uint32_t ov = colhalf ? o[8 + j] : o[j];
                if (t < len)
                    out[(size_t)t * P.H * kDim] = __float2bfloat16_rn(P.scale * __uint_as_float(ov));
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) fused_kernel(Problem P, SeqMap M, int* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzle acts on absolute shared addresses: align the stages to 1024 B
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Smem& S = *reinterpret_cast<Smem*>(base);
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
            mbar_init(&S.full[s], kProdThreads);   // every producer thread
            mbar_init(&S.empty[s], 1);             // one tensor-core commit
        }
        mbar_init(&S.uo_done, 1);
        mbar_init(&S.s_done, 1);
        mbar_init(&S.s16_ready, kEpiWarps * 32);
        mbar_init(&S.u16_ready, kEpiWarps * 32);
        mbar_init(&S.epi_done, kEpiWarps * 32);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.a_ready[b], kProdThreads);
            mbar_init(&S.t_ready[b], 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    // rows 16..31 of every slot's T diag(b) operand stay zero
    for (int i = threadIdx.x; i < kRing * 16 * 16 / 2; i += kThreads) {
        const int slot = i / 128, e = i % 128;
        reinterpret_cast<uint32_t*>(S.st[slot].tbt + 16 * 16)[e] = 0u;
    }
    tc::fence_proxy_async_smem();
    if (warp == kMmaWarp) {
        tc::tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = S.tmem_base;

    if (warp < kEpiWarps) {
        epilogue(P, U, S, tmem, warp, lane, err);
        tc::fence_before_sync();
        mbar_arrive(&S.epi_done);
    } else if (warp == kMmaWarp) {
        if (lane == 0) mma_issuer(U, S, tmem, err);
        __syncwarp();
        // free tensor memory once the epilogue is done with it
        const bool ok = mbar_wait(&S.epi_done, 0u, err);
        __syncwarp();
        (void)ok;
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    } else if (warp == kSolveWarp) {
        solve(P, U, S, lane, err);
    } else {
        produce(P, U, S, warp - kProdWarp0, lane, err);
    }
}

bool g_attr_set[64] = {};

}  // namespace

size_t fused_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_fused(const Problem& P, const SeqMap& M, int* err, cudaStream_t s) {
    const size_t smem = fused_smem_bytes();
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
