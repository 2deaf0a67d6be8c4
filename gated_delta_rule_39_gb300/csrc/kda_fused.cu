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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

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
constexpr int kLoadWarp = kProdWarp0 + kProdWarps;   // TMA loads of the raw rows (one lane)
constexpr int kRing = 3;                    // chunk-operand slots
constexpr int kRaw = 4;                     // raw-row slots: chunks in flight from HBM
constexpr int kThreads = (kLoadWarp + 1) * 32;

constexpr int A_LD = 17;
constexpr int TB_LD = 24;     // fp16 per row of T diag(b) (48 B: ldmatrix conflict-free)
constexpr int KG_LD = 24;     // fp16 per row of a warp's K 2^G tile (48 B)
constexpr int T_SBO = 272;    // byte step between 8-row groups of the transposed fp16
                              // 128 x 16 tile (16 bytes past 256 spreads row groups over banks)
constexpr int KD_SBO = 512;   // byte step between 8-row groups of the fp32 128 x 16 tile
constexpr int AQ_SBO = 512;   // same for the fp32 16 x 16 A_qk tile

// tensor-memory columns (one allocation of 512)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0;       // S^T, fp32: two buffers of 128 columns (chunk parity)
constexpr uint32_t TM_UO = 256;    // [U | O] accumulators: three buffers of 32 columns

// One chunk's operands for the tensor-core recurrence (canonical K-major layouts).
// The operands multiplied by the fp32 state or by U are fp32 values rounded to
// tf32 (kind::tf32 MMAs read the state and U straight from tensor memory).
struct Stage {
    float buo[4 * 32 * 32];        // B of [U|O] += S^T [-w; Q 2^G]^T: 32 x 128, 128B swizzle
    float kdt[16 * KD_SBO / 4];    // B of the state update: (K 2^(G_last-G))^T 128 x 16
    float aqk[2 * AQ_SBO / 4];     // B of O += U A_qk^T: A_qk 16 x 16
    __half vt[16 * T_SBO / 2];     // A of u^T = V^T (T diag b)^T: V^T 128 x 16, interleaved
    __half tbt[32 * 16];           // B of the u MMA: rows 0-15 T diag(b), rows 16-31 zero
    float gc[kDim];                // 2^G_last
    unsigned char pad_[1280];      // keep sizeof(Stage) a multiple of 1024
};
static_assert(sizeof(Stage) % 1024 == 0, "stages keep the swizzled tiles 1024-byte aligned");
// One chunk's raw rows of q, k, v, g as the TMA engine writes them: per tensor two
// boxes of 16 rows x 64 channels (128 bytes per row, 128-byte swizzle).
struct RawSlot {
    __nv_bfloat16 x[4][2][kChunk * 64];
};
constexpr uint32_t kRawBytes = sizeof(RawSlot);
static_assert(kRawBytes == 16384, "four tensors x 16 rows x 256 bytes");
struct ProdShared {
    float part[2][kProdWarps][2][kChunk * kChunk]; // [chunk parity][warp][A_kk, A_qk] partials
    __half tb[2][kChunk * TB_LD];                  // T diag(b) per chunk parity
    __half kg[kProdWarps][2][kChunk * KG_LD];      // each warp's K 2^G tile per chunk parity
    float A[kChunk * A_LD];                        // solver scratch
};
struct Smem {
    Stage st[kRing];
    RawSlot raw[kRaw];
    ProdShared pr;
    unsigned long long raw_full[kRaw];   // TMA bytes landed
    unsigned long long raw_empty[kRaw];  // producers have read the slot
    unsigned long long full[kRing];    // producers -> MMA / epilogue
    unsigned long long empty[kRing];   // MMA commit -> producers
    unsigned long long a_ready[2];     // producers' partial A_kk / A_qk summed
    unsigned long long t_ready[2];     // solver: T diag(b), A_qk written
    unsigned long long uo_done;        // U|O MMAs complete
    unsigned long long s_done;         // state update + O MMAs complete
    unsigned long long init_ready;     // epilogue: initial state written
    unsigned long long scaled;         // epilogue: 2^G_last S^T written to the other buffer
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
__device__ __forceinline__ float2 bf2_to_f2(uint32_t raw) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&raw);
    return __bfloat1622float2(v);
}
__device__ __forceinline__ float tf32_round(float x) { return __uint_as_float(to_tf32(x)); }

struct Unit {
    int n, h, tok_start, L, nch;
};

// ---- raw-row loads on the TMA engine (one thread) ----------------------------------
// Tensor maps over q, k, v, g viewed as [rows][H][128] bf16 (rows = B*T tokens).
// Rows past the end of the tensor are zero-filled; rows past the end of a
// sequence belong to the next one and are masked by the producers.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

__device__ void loader(const RawMaps& TM, const Unit& U, Smem& S, int* err) {
    const CUtensorMap* maps[4] = {&TM.q, &TM.k, &TM.v, &TM.g};
    for (int c = 0; c < U.nch; ++c) {
        const int slot = c % kRaw;
        if (c >= kRaw && !mbar_wait(&S.raw_empty[slot], (unsigned)(((c / kRaw) - 1) & 1), err))
            break;
        const uint32_t full = smem_u32(&S.raw_full[slot]);
        tc::mbar_arrive_expect_tx(full, kRawBytes);
        const int row = U.tok_start + c * kChunk;
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tma_load_3d(smem_u32(S.raw[slot].x[t][half]), maps[t], 64 * half, U.h, row, full);
    }
    // do not let the CTA exit while copies it issued are still landing
    const int first = U.nch > kRaw ? U.nch - kRaw : 0;
    for (int c = first; c < U.nch; ++c)
        if (!mbar_wait(&S.raw_full[c % kRaw], (unsigned)((c / kRaw) & 1), err)) break;
}

// ---- token-parallel stage: producer warp w, channels 16w .. 16w+15 ----------------
// Lane (g, t) = (lane >> 2, lane & 3) holds rows g and g+8 of the chunk for the
// channel pairs p = 16w + 8kk + 2t, p+1 (kk = 0, 1).  In the tf32 MMA fragments
// of k-step kk the pair plays logical columns t and t+4; the decay-ratio
// products sum over channels, so this relabelling leaves them unchanged.
struct RawSlice {
    uint32_t q[2][2], k[2][2], v[2][2], g[2][2];   // [row g / g+8][kk] bf16 pairs
};

__device__ __forceinline__ void lds_slice(const RawSlot& R, int w, int lg, int lt, int len,
                                          RawSlice& X) {
    const int half = w >> 2;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = lg + 8 * i;
        const bool ok = r < len;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int chunk16 = 2 * (w & 3) + kk;   // 16-byte chunk of the 128-byte row
            const int off = r * 128 + ((chunk16 ^ (r & 7)) << 4) + 4 * lt;
            const auto ld = [&](int t) {
                return ok ? *reinterpret_cast<const uint32_t*>(
                                reinterpret_cast<const unsigned char*>(R.x[t][half]) + off)
                          : 0u;
            };
            X.q[i][kk] = ld(0);
            X.k[i][kk] = ld(1);
            X.v[i][kk] = ld(2);
            X.g[i][kk] = ld(3);
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

    for (int c = 0; c <= U.nch; ++c) {
        if (c < U.nch) {
            const int len = min(kChunk, U.L - c * kChunk);
            const int rslot = c % kRaw;
            bool ok = mbar_wait(&S.raw_full[rslot], (unsigned)((c / kRaw) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return;
            RawSlice X;
            lds_slice(S.raw[rslot], w, lg, lt, len, X);
            mbar_arrive(&S.raw_empty[rslot]);   // release: the reads above come first
            const int slot = c % kRing;
            Stage& st = S.st[slot];
            const int par = c & 1;
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
                    *reinterpret_cast<float2*>(buo + tc::swizzled32_offset(16 + r, p, 32)) =
                        make_float2(__uint_as_float(aqf[kk][i]), __uint_as_float(aqf[kk][i + 2]));
                    *reinterpret_cast<uint32_t*>(&kgt[r * KG_LD + 8 * kk + 2 * lt]) =
                        pack_half2(kg0, kg1);
                    *reinterpret_cast<float*>(kdt + tc::interleaved32_offset(p, r, KD_SBO)) =
                        tf32_round(kd.x);
                    *reinterpret_cast<float*>(kdt + tc::interleaved32_offset(p + 1, r, KD_SBO)) =
                        tf32_round(kd.y);
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
            *reinterpret_cast<float2*>(buo + tc::swizzled32_offset(lg, col0, 32)) =
                make_float2(tf32_round(-cw0[0]), tf32_round(-cw0[1]));
            *reinterpret_cast<float2*>(buo + tc::swizzled32_offset(lg + 8, col0, 32)) =
                make_float2(tf32_round(-cw0[2]), tf32_round(-cw0[3]));
            *reinterpret_cast<float2*>(buo + tc::swizzled32_offset(lg, col1, 32)) =
                make_float2(tf32_round(-cw1[0]), tf32_round(-cw1[1]));
            *reinterpret_cast<float2*>(buo + tc::swizzled32_offset(lg + 8, col1, 32)) =
                make_float2(tf32_round(-cw1[2]), tf32_round(-cw1[3]));
            // generic-proxy writes of this thread -> visible to the tensor core
            tc::fence_proxy_async_smem();
            mbar_arrive(&S.full[cp % kRing]);
        }
    }
}

// ---- solver warp: (I + A_kk)^-1, T diag(b), A_qk for every chunk ------------------
__device__ void solve(const Problem& P, const Unit& U, Smem& S, int lane, int* err) {
    ProdShared& PS = S.pr;
    // beta logits in windows of 64 tokens (4 chunks), the next window loaded one
    // window ahead: lane i holds tokens 64 j + i and 64 j + 32 + i of window j
    const __nv_bfloat16* beta = P.beta + (size_t)U.tok_start * P.H + U.h;
    const auto load_window = [&](int j, float& w0, float& w1) {
        const int t0 = 64 * j + lane, t1 = t0 + 32;
        w0 = (t0 < U.L) ? __bfloat162float(beta[(size_t)t0 * P.H]) : 0.0f;
        w1 = (t1 < U.L) ? __bfloat162float(beta[(size_t)t1 * P.H]) : 0.0f;
    };
    float bw0 = 0.0f, bw1 = 0.0f, nb0 = 0.0f, nb1 = 0.0f;
    if (U.nch > 0) load_window(0, nb0, nb1);
    for (int c = 0; c < U.nch; ++c) {
        const int len = min(kChunk, U.L - c * kChunk);
        if ((c & 3) == 0) {
            bw0 = nb0;
            bw1 = nb1;
            if (64 * (c / 4 + 1) < U.L) load_window(c / 4 + 1, nb0, nb1);
        }
        const float lw = __shfl_sync(0xffffffffu, (c & 2) ? bw1 : bw0, 16 * (c & 1) + (lane & 15));
        const float bl = (lane < len) ? sigmoid_fast(lw) : 0.0f;   // b of row `lane`
        const int par = c & 1;
        const bool ok = mbar_wait(&S.a_ready[par], (unsigned)((c >> 1) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return;
        Stage& st = S.st[c % kRing];
        // A_kk = diag(b) (sum of the warps' partials), strictly lower; A_qk inclusive
        // lower (tf32, interleaved); partials summed in warp order
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
            *reinterpret_cast<float2*>(reinterpret_cast<unsigned char*>(st.aqk) +
                                       tc::interleaved32_offset(r, s, AQ_SBO)) =
                make_float2((s <= r) ? tf32_round(sq.x) : 0.0f, (s + 1 <= r) ? tf32_round(sq.y) : 0.0f);
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
// Per chunk c (slot s), in the transposed orientation (TMEM lane = value row v), with
// S^T of the chunk's start in state buffer c & 1:
//   [U|O] = V^T [T diag(b) ; 0]^T             (u^T into the U half, zeros into O; fp16)
//   [U|O] += S^T [-w ; Q 2^G]^T               (16 tf32 MMAs over the 128 key channels)
//   S'^T += U^T (K 2^(G_last-G))              (S'^T = S^T 2^G_last, written by the
//                                              epilogue into the other state buffer)
//   O    += U^T A_qk^T
// The state and U are read from tensor memory as fp32 A operands (kind::tf32).
__device__ void mma_issuer(const Unit& U, Smem& S, uint32_t tmem, int* err) {
    constexpr uint32_t id_u = tc::idesc_f16_f32(128, 32);
    constexpr uint32_t id_s = tc::idesc_tf32_f32(128, 32);
    constexpr uint32_t id_k = tc::idesc_tf32_f32(128, 128);
    constexpr uint32_t id_q = tc::idesc_tf32_f32(128, 16);
    // descriptors of slot 0; slot s adds its byte offset >> 4 to the start field
    const uint64_t d_vt = tc::smem_desc(smem_u32(S.st[0].vt), 128, T_SBO, tc::kSwizzleNone);
    const uint64_t d_tbt = tc::smem_desc(smem_u32(S.st[0].tbt), 128, 256, tc::kSwizzleNone);
    const uint64_t d_buo = tc::smem_desc(smem_u32(S.st[0].buo), 16, 1024, tc::kSwizzle128B);
    const uint64_t d_kdt = tc::smem_desc(smem_u32(S.st[0].kdt), 128, KD_SBO, tc::kSwizzleNone);
    const uint64_t d_aqk = tc::smem_desc(smem_u32(S.st[0].aqk), 128, AQ_SBO, tc::kSwizzleNone);
    for (int c = 0; c < U.nch; ++c) {
        const int slot = c % kRing;
        const uint64_t so = (uint64_t)((slot * sizeof(Stage)) >> 4);
        const uint32_t sc = tmem + TM_S + 128u * (c & 1);
        const uint32_t sn = tmem + TM_S + 128u * ((c + 1) & 1);
        const uint32_t uo = tmem + TM_UO + 32u * (c % 3);
        if (!mbar_wait(&S.full[slot], (unsigned)((c / kRing) & 1), err)) return;
        if (c == 0) {
            if (!mbar_wait(&S.init_ready, 0u, err)) return;
        } else {
            if (!mbar_wait(&S.s_done, (unsigned)((c - 1) & 1), err)) return;
        }
        tc::fence_after_sync();
        tc::mma_ss(uo, d_vt + so, d_tbt + so, id_u, 0);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            tc::mma_ts_tf32(uo, sc + 8 * kk,
                            d_buo + so + (uint64_t)(((kk >> 2) * 4096 + (kk & 3) * 32) >> 4), id_s, 1);
        tc::commit(smem_u32(&S.uo_done));
        if (!mbar_wait(&S.uo_done, (unsigned)(c & 1), err)) return;
        if (!mbar_wait(&S.scaled, (unsigned)(c & 1), err)) return;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            tc::mma_ts_tf32(sn, uo + 8 * kk, d_kdt + so + (uint64_t)((kk * 256) >> 4), id_k, 1);
            tc::mma_ts_tf32(uo + 16, uo + 8 * kk, d_aqk + so + (uint64_t)((kk * 256) >> 4), id_q, 1);
        }
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
// owns half of the state's columns (key channels 64 (ew / 4) .. + 63) and the
// outputs of tokens 8 (ew / 4) .. + 7.  Once the state of chunk c's start is
// complete, it writes 2^G_last(c) times it into the other state buffer, which the
// update MMAs of chunk c accumulate into while the U|O MMAs still read the first.
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
    // initial state S0 into buffer 0, then S0 Diag(2^G_last of chunk 0) into buffer 1
#pragma unroll 1
    for (int piece = p0; piece < p0 + 2; ++piece) {
        uint32_t x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = 32 * piece + i;
            x[i] = __float_as_uint(P.init_state ? state_in(P, sbase + (size_t)c * kDim) : 0.0f);
        }
        tc::st32(tl + TM_S + 32 * piece, x);
    }
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(&S.init_ready);
    ok = mbar_wait(&S.full[0], 0u, err);
    if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll 1
    for (int piece = p0; piece < p0 + 2; ++piece) {
        uint32_t x[32];
        tc::ld32(tl + TM_S + 32 * piece, x);
        tc::wait_ld();
        scale32(x, S.st[0].gc + 32 * piece);
        tc::st32(tl + TM_S + 128 + 32 * piece, x);
    }
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(&S.scaled);

    for (int c = 1; c <= U.nch; ++c) {
        // chunk c - 1 finished: its end state is in buffer c & 1
        ok = mbar_wait(&S.s_done, (unsigned)((c - 1) & 1), err);
        const bool more = c < U.nch;
        const int slot = c % kRing;
        if (more) ok = ok && mbar_wait(&S.full[slot], (unsigned)((c / kRing) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc::fence_after_sync();
        const uint32_t sc = tl + TM_S + 128u * (c & 1);
        if (more) {
            const uint32_t sn = tl + TM_S + 128u * ((c + 1) & 1);
#pragma unroll 1
            for (int piece = p0; piece < p0 + 2; ++piece) {
                uint32_t x[32];
                tc::ld32(sc + 32 * piece, x);
                tc::wait_ld();
                scale32(x, S.st[slot].gc + 32 * piece);
                tc::st32(sn + 32 * piece, x);
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(&S.scaled);
        } else if (P.final_state) {
#pragma unroll 1
            for (int piece = p0; piece < p0 + 2; ++piece) {
                uint32_t x[32];
                tc::ld32(sc + 32 * piece, x);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    state_out(P, sbase + (size_t)(32 * piece + i) * kDim, __uint_as_float(x[i]));
            }
        }
        // outputs of chunk c - 1, tokens 8 colhalf .. + 7: O^T lane v, column t
        {
            const int cp = c - 1;
            uint32_t o[16];
            tc::ld16(tl + TM_UO + 32u * (cp % 3) + 16, o);
            tc::wait_ld();
            const int len = min(kChunk, U.L - cp * kChunk);
            __nv_bfloat16* out = P.out + ((size_t)(U.tok_start + cp * kChunk) * P.H + U.h) * kDim + v;
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

__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(Problem P, SeqMap M, const __grid_constant__ RawMaps TM, int* err) {
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
        mbar_init(&S.init_ready, kEpiWarps * 32);
        mbar_init(&S.scaled, kEpiWarps * 32);
        mbar_init(&S.epi_done, kEpiWarps * 32);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.a_ready[b], kProdThreads);
            mbar_init(&S.t_ready[b], 32);
        }
        for (int s = 0; s < kRaw; ++s) {
            mbar_init(&S.raw_full[s], 1);                 // loader's arrive + TMA bytes
            mbar_init(&S.raw_empty[s], kProdThreads);     // every producer thread
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
    } else if (warp == kLoadWarp) {
        if (lane == 0) loader(TM, U, S, err);
    } else {
        produce(P, U, S, warp - kProdWarp0, lane, err);
    }
}

bool g_attr_set[64] = {};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// [rows][H][128] bf16 viewed as a 3-D tensor (channel, head, row); boxes of
// 64 channels x 1 head x 16 rows, 128-byte swizzle (one 128-byte row per token)
cudaError_t encode_rows(CUtensorMap* map, const void* base, int H, long long rows) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)H, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)H * kDim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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
    // total token rows: B*T (fixed length, N = B sequences of T) or T (varlen, B = 1)
    const long long rows = (P.cu_seqlens == nullptr) ? (long long)P.N * P.T : (long long)P.T;
    RawMaps TM;
    if (rows > 0) {
        cudaError_t e = encode_rows(&TM.q, P.q, P.H, rows);
        if (e == cudaSuccess) e = encode_rows(&TM.k, P.k, P.H, rows);
        if (e == cudaSuccess) e = encode_rows(&TM.v, P.v, P.H, rows);
        if (e == cudaSuccess) e = encode_rows(&TM.g, P.g, P.H, rows);
        if (e != cudaSuccess) return e;
    } else {
        memset(&TM, 0, sizeof(TM));   // no tokens: the loader issues nothing
    }
    fused_kernel<<<(unsigned)ctas, kThreads, smem, s>>>(P, M, TM, err);
    return cudaGetLastError();
}

}  // namespace kda
