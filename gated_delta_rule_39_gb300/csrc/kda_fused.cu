// Fused KDA forward kernel: one CTA per (sequence, head) runs both stages of
// the chunkwise algorithm, so q, k, v, g and beta are read from HBM once and
// only the output and the states are written.
//
//   loader warp         TMA tensor loads of each chunk's raw q, k, v, g rows into a
//                       ring of shared-memory slots, several chunks ahead.
//   producer warps (8)  the token-parallel stage.  Warp w owns key / value channels
//                       16w .. 16w+15; each thread holds one channel pair over four
//                       consecutive rows of the 16-token chunk.  They compute the
//                       gates, the in-chunk cumulative base-2 log-decay G, the decay
//                       factors and the operand tiles of the chunk (K 2^G, Q 2^G,
//                       K 2^-G, K 2^(G_last-G), V), up to kRing chunks ahead.
//   A-product warps (2) the decay-ratio products A_kk = (K 2^G)(K 2^-G)^T (to the
//                       solver) and A_qk = (Q 2^G)(K 2^-G)^T (inclusive lower, to
//                       an operand tile, which completes the stage with -w): tf32
//                       mma.sync from ldmatrix fragments.
//   w warps (2)         once the solver has T: -w = -T diag(b)(K 2^G), 64 channels
//                       each, which completes the chunk's operands.
//   solver warp         T = (I + diag(b) A_kk)^-1 as a four-factor Neumann product
//                       (fp16 mma.sync), then T diag(b).
//   MMA warp            issues the tcgen05 MMAs of the recurrence (one thread).
//   epilogue warps (4)  own the tensor-memory state S^T (lane v = value channel v):
//                       decay rescale, outputs, initial and final state.
//
// Chunkwise DPLR-variant (WY) algorithm with 16-token chunks, a 16 x 16
// inverse and base-2 gates: "Moonshot AI Open-Sources FlashKDA", sections
// "Why KDA?" and "What makes the kernel fast".  The pages split the two
// stages into two kernels on Hopper because the sequential stage alone left
// SMs idle; here the split stays, but inside one CTA, so the intermediate
// factors never leave the SM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_tcgen05.cuh"

// Every wait of the kernel is bounded.  A pipeline wait gives up after KDA_SPIN_LIMIT
// SM cycles (about 2 s at the default): it records KDA_ERR_DEVICE_TIMEOUT in the error
// word and its role stops.  Before a CTA exits, the roles that started asynchronous work
// wait for it (up to KDA_DRAIN_LIMIT cycles each): the loader for the TMA copies it
// issued, the MMA thread for its MMAs and commits; tensor memory is released only after
// the MMA thread has drained and the epilogue has finished with it.  Both limits can be
// set at build time (-DKDA_SPIN_LIMIT=...).
#ifndef KDA_SPIN_LIMIT
#define KDA_SPIN_LIMIT (1LL << 32)
#endif
#ifndef KDA_DRAIN_LIMIT
#define KDA_DRAIN_LIMIT (1LL << 33)
#endif

namespace kda {

namespace {

constexpr int kEpiWarps = 4;                // epilogue: one warp per TMEM lane quarter
constexpr int kProdWarps = 8;               // 16 key channels each
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kRing = 4;                    // chunk-operand slots (live until the recurrence is done)
constexpr int kEarly = 2;                   // K 2^G / K 2^-G slots (live until the products are done)
constexpr int kRaw = 3;                     // raw-row slots: chunks in flight from HBM

// Warp roles.  A warp's SM sub-partition (scheduler) is its index mod 4, so the
// placement decides which roles share issue slots; the producers (most of the
// instructions) are spread two per sub-partition.  Epilogue warp q must have
// index = q (mod 4) to reach TMEM lanes 32q .. 32q + 31.
enum Role : uint8_t { kEpi, kSolve, kAprod0, kAprod1, kW0, kW1, kMma, kProd, kLoad };
constexpr int kNumWarps = 19;
constexpr int kThreads = kNumWarps * 32;
__host__ __device__ constexpr Role role_of(int warp) {
    switch (warp) {
        case 0: case 1: case 2: case 3: return kEpi;   // lane quarters 0-3
        case 4: return kSolve;                          // sub-partition 0
        case 5: return kW0;                             // 1
        case 6: return kAprod1;                         // 2
        case 7: return kAprod0;                         // 3 (the only single-warp role there)
        case 8: return kW1;                             // 0
        case 9: return kMma;                            // 1
        case 18: return kLoad;                          // 2
        default: return kProd;                          // 10-17: two per sub-partition
    }
}
// producer slice of warp i: its rank among the producer warps
__host__ __device__ constexpr int prod_index(int warp) {
    int n = 0;
    for (int i = 0; i < warp; ++i) n += role_of(i) == kProd;
    return n;
}
__host__ __device__ constexpr int count_role(Role r) {
    int n = 0;
    for (int i = 0; i < kNumWarps; ++i) n += role_of(i) == r;
    return n;
}
__host__ __device__ constexpr int find_role(Role r) {
    for (int i = 0; i < kNumWarps; ++i)
        if (role_of(i) == r) return i;
    return -1;
}
static_assert(count_role(kProd) == kProdWarps && count_role(kEpi) == kEpiWarps, "role table");
static_assert(count_role(kSolve) == 1 && count_role(kMma) == 1 && count_role(kLoad) == 1 &&
              count_role(kAprod0) == 1 && count_role(kAprod1) == 1 && count_role(kW0) == 1 &&
              count_role(kW1) == 1, "role table");
static_assert(role_of(0) == kEpi && role_of(1) == kEpi && role_of(2) == kEpi && role_of(3) == kEpi,
              "epilogue warps 0-3 own lane quarters 0-3");
constexpr int kMmaWarp = find_role(kMma);

constexpr int AK_LD = 20;     // fp32 per row of A_kk handed to the solver (16-byte rows)
constexpr int TB_LD = 24;     // fp16 per row of T diag(b) (48 B: ldmatrix conflict-free)
constexpr int T_SBO = 256;    // byte step between 8-row groups of the transposed fp16 128 x 16 tile
constexpr int KD_SBO = 528;   // same for the fp32 128 x 16 tile
constexpr int AQ_SBO = 512;   // fp32 16 x 16 A_qk tile
constexpr int X_ROWS = 32;    // rows of the [Q 2^G ; -w] tile

// tensor-memory columns (one allocation of 512)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0;       // S^T, fp32: two buffers of 128 columns (chunk parity)
constexpr uint32_t TM_UO = 256;    // [O | U] accumulators: three buffers of 32 columns

// One chunk's operands for the tensor-core recurrence (canonical K-major layouts).
// The operands multiplied by the fp32 state or by U are fp32 values rounded to
// tf32 (kind::tf32 MMAs read the state and U straight from tensor memory).
struct Stage {
    // rows 0-15 Q 2^G, rows 16-31 -w; 128 key channels; 128B swizzle, [K block of 32
    // channels][32 rows][128 bytes]: the B operand of [O|U] += S^T [Q 2^G ; -w]^T
    float x[4 * X_ROWS * 32];
    float kdt[16 * KD_SBO / 4];    // B of the state update: (K 2^(G_last-G))^T 128 x 16
    float aqk[2 * AQ_SBO / 4];     // B of O += U A_qk^T: A_qk 16 x 16
    __half vt[16 * T_SBO / 2];     // A of u^T = V^T (T diag b)^T: V^T 128 x 16, interleaved
    __half tbt[16 * 16];           // B of the u MMA: T diag(b), 16 x 16, interleaved
    float gc[kDim];                // 2^G_last
    __half kgh[kChunk * kDim];     // K 2^G in fp16, [token][channel] (kgh_offset): B of w
    __half tbr[kChunk * TB_LD];    // T diag(b) fp16 row-major: A of w
};
// K 2^G and K 2^-G (tf32, [K block][16 rows][128 bytes], 128B swizzle): read only by
// the decay-ratio products, so they live in a shorter ring than the operand stages.
struct EarlySlot {
    float kg[4 * kChunk * 32];
    float ki[4 * kChunk * 32];
};
static_assert(sizeof(Stage) % 1024 == 0, "stages keep the swizzled tiles 1024-byte aligned");
// fp16 K 2^G tile: 256-byte rows, 16-byte chunks XOR-swizzled by row % 8 so that the
// eight rows an ldmatrix reads fall in distinct banks.  Byte offset of (row, col).
__device__ __forceinline__ int kgh_offset(int row, int col) {
    return row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2;
}

// One chunk's raw rows of q, k, v, g as the TMA engine writes them: per tensor two
// boxes of 16 rows x 64 channels (128 bytes per row, 128-byte swizzle).
struct RawSlot {
    __nv_bfloat16 x[4][2][kChunk * 64];
};
constexpr uint32_t kRawBytes = sizeof(RawSlot);
static_assert(kRawBytes == 16384, "four tensors x 16 rows x 256 bytes");
struct ProdShared {
    float Akk[2][kChunk * AK_LD];                  // A_kk (before diag(b)) per chunk parity
};
constexpr int kUnitRing = 8;   // unit indices the loader may publish ahead of the roles
// warps that read each published unit index: epilogue 4, MMA 1, solver 1, A products 2,
// w 2, producers 8 (every warp but the loader's)
constexpr int kUnitReaders = 18;

struct Smem {
    Stage st[kRing];
    EarlySlot early[kEarly];
    RawSlot raw[kRaw];
    ProdShared pr;
    unsigned long long raw_full[kRaw];   // TMA bytes landed
    unsigned long long raw_empty[kRaw];  // producers have read the slot
    unsigned long long full[kRing];      // operands complete (-w, A_qk written) -> MMA / epilogue
    unsigned long long empty[kRing];     // MMA commit -> producers
    unsigned long long kq_ready[kRing];  // producers: the chunk's tiles written
    unsigned long long a_ready[2];       // A_kk warp: A_kk written (per chunk parity)
    unsigned long long t_ready[kRing];   // solver: T diag(b) written
    unsigned long long e_free[kEarly];   // both A-product warps are done with the early slot
    unsigned long long s_done;           // state update + O MMAs complete
    unsigned long long init_ready;       // epilogue: initial state written
    unsigned long long scaled;           // epilogue: 2^G_last S^T written to the other buffer,
                                         // and the chunk's O|U MMAs complete (commit)
    unsigned long long epi_done;         // epilogue finished with tensor memory
    unsigned long long drain;            // the MMA thread's exit drain (one commit)
    // persistent calls: the units this CTA takes, in order (loader -> every role)
    unsigned long long unit_full[kUnitRing];    // the loader wrote unit[slot]
    unsigned long long unit_empty[kUnitRing];   // every consumer warp has read it
    int unit[kUnitRing][6];                     // n, h, tok_start, L, nch (-1: none), vzero
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
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)   // suspends for a system-dependent time limit
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` SM cycles and reports a timeout.
__device__ __forceinline__ bool mbar_wait(unsigned long long* b, unsigned parity, int* err,
                                          long long limit = KDA_SPIN_LIMIT) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > limit) {
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
__device__ __forceinline__ float2 f2add(float2 a, float2 b) {
    unsigned long long x, y, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("add.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(z));
    return r;
}
__device__ __forceinline__ float2 f2sub(float2 a, float2 b) {
    unsigned long long x, y, z;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("sub.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(z));
    return r;
}
__device__ __forceinline__ uint32_t pack_halves(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t raw) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&raw);
    return __bfloat1622float2(v);
}
// fp32 -> tf32 operand, rounded to nearest with ties away from zero.  The default
// adds half a tf32 ulp to the bit pattern and leaves the 13 low bits for the tensor
// core to drop: its tf32 operands read only the top 19 bits of an fp32 register or
// shared-memory word (measured: whole-call results are bit-identical to those of
// the build with -DKDA_TF32_CVT, which rounds with cvt.rna.tf32.f32 and clears the
// low bits; a GPU test compares the two builds).  The addition is one instruction
// where the conversion makes the whole call 14 % slower (0.680 against 0.599 ms on
// T = 8192, H = 96).
__device__ __forceinline__ float tf32_round(float x) {
#ifdef KDA_TF32_CVT
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return __uint_as_float(y);
#else
    return __uint_as_float(__float_as_uint(x) + 0x1000u);
#endif
}

struct Unit {
    int n, h, tok_start, L, nch;   // n: index of the initial and final state
    bool vzero;                    // values taken as zero (v read from 16 zero rows)
};

// Unit `id` of a launch (id = rank * H + h): its head, tokens and state index.
__device__ __forceinline__ Unit unit_at(const Problem& P, const SeqMap& M, int id) {
    Unit U;
    U.h = id % P.H;
    const int rank = id / P.H;
    U.vzero = false;
    if (P.window >= 0) {
        // sequence split (fixed length): the unit's sequence, segment and kind.  Its
        // initial state (prepared on the host side: the caller's, zero or identity) and
        // its final state are at index rank of fp32 scratch.
        const int per = P.window == 0 ? 2 * P.nseg - 3 : P.nseg - 1;
        const int seq = rank / per, vj = rank % per;
        int j = P.window == 0 ? vj : vj + 1;      // segment
        if (P.window == 0 && vj > P.nseg - 2) {
            j = vj - (P.nseg - 2);                // transition operator: zero values
            U.vzero = true;
        }
        U.n = rank;
        const long long nchk = (P.T + kChunk - 1) / kChunk;
        const int c0 = (int)((long long)j * nchk / P.nseg);
        const int c1 = (int)((long long)(j + 1) * nchk / P.nseg);
        U.tok_start = seq * P.T + c0 * kChunk;
        U.L = min(c1 * kChunk, P.T) - c0 * kChunk;
    } else if (P.cu_seqlens == nullptr) {
        U.n = rank;
        U.tok_start = rank * P.T;
        U.L = P.T;
    } else {
        U.n = M.seq_order[rank];
        U.tok_start = P.cu_seqlens[U.n];
        U.L = P.cu_seqlens[U.n + 1] - U.tok_start;
    }
    U.nch = (U.L + kChunk - 1) / kChunk;
    return U;
}

// Persistent calls: the CTA's k-th unit.  The loader takes the next unit of the whole
// launch from a device counter (units in longest-first order, so this is list
// scheduling, longest first), decodes it and publishes it in slot k of the unit ring;
// every other warp copies it from there, so no role reads the sequence map itself.  A
// slot is free again once every reader has copied it, so the loader can run at most
// kUnitRing units ahead of the slowest role's current unit.  nch = -1: no more units.
__device__ bool publish_unit(const Problem& P, const SeqMap& M, Smem& S, int k, int* err, Unit& U) {
    const int slot = k % kUnitRing;
    if (k >= kUnitRing &&
        !mbar_wait(&S.unit_empty[slot], (unsigned)(((k / kUnitRing) - 1) & 1), err))
        return false;
    const int id = atomicAdd(M.counter, 1);
    if (id < P.N * P.H) {
        U = unit_at(P, M, id);
    } else {
        U = Unit{};
        U.nch = -1;
    }
    volatile int* w = S.unit[slot];
    w[0] = U.n;
    w[1] = U.h;
    w[2] = U.tok_start;
    w[3] = U.L;
    w[4] = U.nch;
    w[5] = U.vzero;
    mbar_arrive(&S.unit_full[slot]);   // release: the unit is visible to the readers
    return U.nch >= 0;
}
// A reader's k-th unit; false: none, or a wait gave up.  whole_warp: all 32 lanes call it
// and lane 0 releases the slot; otherwise the one calling thread does.
__device__ bool read_unit(Smem& S, int k, int* err, bool whole_warp, Unit& U) {
    const int slot = k % kUnitRing;
    bool ok = mbar_wait(&S.unit_full[slot], (unsigned)((k / kUnitRing) & 1), err);
    if (whole_warp) ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    const volatile int* r = S.unit[slot];
    U.n = r[0];
    U.h = r[1];
    U.tok_start = r[2];
    U.L = r[3];
    U.nch = r[4];
    U.vzero = r[5] != 0;
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(&S.unit_empty[slot]);
    return U.nch >= 0;
}

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

// One unit's chunks; g0 = this CTA's chunks before it (ring slots and barrier phases
// continue across the units of a persistent CTA).  Returns the chunks issued.
__device__ __forceinline__ int loader_unit(const RawMaps& TM, const Unit& U, Smem& S, int* err,
                                           int g0) {
    const CUtensorMap* maps[4] = {&TM.q, &TM.k, U.vzero ? &TM.vz : &TM.v, &TM.g};
    int c = 0;   // chunks issued
    for (; c < U.nch; ++c) {
        const int g = g0 + c;
        const int slot = g % kRaw;
        if (g >= kRaw && !mbar_wait(&S.raw_empty[slot], (unsigned)(((g / kRaw) - 1) & 1), err))
            break;
        const uint32_t full = smem_u32(&S.raw_full[slot]);
        tc::mbar_arrive_expect_tx(full, kRawBytes);
        const int row = U.tok_start + c * kChunk;
        const int vrow = U.vzero ? 0 : row;   // zero values: the same 16 zero rows each chunk
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tma_load_3d(smem_u32(S.raw[slot].x[t][half]), maps[t], 64 * half, U.h,
                            t == 2 ? vrow : row, full);
    }
    return c;
}

template <bool kP>
__device__ void loader(const Problem& P, const SeqMap& M, const RawMaps& TM, const Unit& U0,
                       Smem& S, int* err) {
    int n = 0;   // chunks issued
    if constexpr (!kP) {
        n = loader_unit(TM, U0, S, err, 0);
    } else {
        for (int k = 0;; ++k) {
            Unit U;
            if (!publish_unit(P, M, S, k, err, U)) break;
            const int done = loader_unit(TM, U, S, err, n);
            n += done;
            if (done < U.nch) break;   // a wait gave up
        }
    }
    // Do not let the CTA exit while copies it issued are still landing.  Each slot has at
    // most one copy in flight (the next one waits for raw_empty), so the last issues of
    // the slots are the only phases that may be pending; also after a wait gave up.
    const int first = n > kRaw ? n - kRaw : 0;
    for (int i = first; i < n; ++i)
        mbar_wait(&S.raw_full[i % kRaw], (unsigned)((i / kRaw) & 1), err, KDA_DRAIN_LIMIT);
}

// ---- token-parallel stage: producer warp w, channels 16w .. 16w+15 ----------------
// Lane (pi, j) = (lane & 7, lane >> 3) holds channels c0 = 16w + 2 pi, c0 + 1 over rows
// 4j .. 4j+3 of the chunk.
// One unit's chunks (g0 as for the loader); false if a wait gave up.
__device__ __forceinline__ bool produce_unit(const Problem& P, const Unit& U, Smem& S, int w, int lane,
                                             int* err, int g0) {
    const int pi = lane & 7, j = lane >> 3;
    const int c0 = 16 * w + 2 * pi;
    const int r0 = 4 * j;
    const float expA = expf(P.A_log[U.h]);
    const float ga = -expA * kLog2e;   // sigmoid argument in base 2: g ga + gb
    const float2 gb = make_float2(ga * P.dt_bias[(size_t)U.h * kDim + c0],
                                  ga * P.dt_bias[(size_t)U.h * kDim + c0 + 1]);
    const float lb2 = P.lower_bound * kLog2e;
    // raw-slot addressing: box (channel half), 16-byte chunk of the 128-byte row, offset
    const int half = w >> 2;
    const int chunk16 = 2 * (w & 3) + (pi >> 2);
    const int inoff = 4 * (pi & 3);
    for (int c = 0; c < U.nch; ++c) {
        const int g = g0 + c;
        {
            const int len = min(kChunk, U.L - c * kChunk);
            const int rslot = g % kRaw;
            bool ok = mbar_wait(&S.raw_full[rslot], (unsigned)((g / kRaw) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return false;
            uint32_t rq[4], rk[4], rv[4], rg[4];
            {
                const RawSlot& R = S.raw[rslot];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = r0 + i;
                    const bool in = r < len;
                    const int off = r * 128 + ((chunk16 ^ (r & 7)) << 4) + inoff;
                    const auto ld = [&](int t) {
                        return in ? *reinterpret_cast<const uint32_t*>(
                                        reinterpret_cast<const unsigned char*>(R.x[t][half]) + off)
                                  : 0u;
                    };
                    rq[i] = ld(0);
                    rk[i] = ld(1);
                    rv[i] = ld(2);
                    rg[i] = ld(3);
                }
            }
            // The slot's next writer is the TMA engine (async proxy): order this
            // thread's generic-proxy reads before it, then release the slot.
            tc::fence_proxy_async_smem();
            mbar_arrive(&S.raw_empty[rslot]);
            const int slot = g % kRing;
            Stage& st = S.st[slot];
            if (g >= kRing) ok = mbar_wait(&S.empty[slot], (unsigned)(((g / kRing) - 1) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return false;

            // gates lower_bound * sigmoid(exp(A_log) (g + dt_bias)), base 2; rows past the
            // sequence end decay by nothing
            float2 G[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 xa = f2fma(bf2_to_f2(rg[i]), make_float2(ga, ga), gb);
                const float2 sg = f2mul(make_float2(rcp_approx(1.0f + ex2_approx(xa.x)),
                                                    rcp_approx(1.0f + ex2_approx(xa.y))),
                                        make_float2(lb2, lb2));
                G[i] = (r0 + i < len) ? sg : make_float2(0.0f, 0.0f);
            }
            // inclusive cumulative sum over the 16 rows: within the thread's four rows,
            // then across the four row groups (lanes 8 apart)
            G[1] = f2add(G[1], G[0]);
            G[2] = f2add(G[2], G[1]);
            G[3] = f2add(G[3], G[2]);
            float2 incl = G[3];
#pragma unroll
            for (int d = 8; d < 32; d <<= 1) {
                const float2 y = make_float2(__shfl_up_sync(0xffffffffu, incl.x, d),
                                             __shfl_up_sync(0xffffffffu, incl.y, d));
                if (lane >= d) incl = f2add(incl, y);
            }
            const float2 excl = f2sub(incl, G[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) G[i] = f2add(G[i], excl);
            const float2 glast = make_float2(__shfl_sync(0xffffffffu, incl.x, 24 + pi),
                                             __shfl_sync(0xffffffffu, incl.y, 24 + pi));
            const float2 gc = make_float2(ex2_approx(glast.x), ex2_approx(glast.y));
            if (j == 0) *reinterpret_cast<float2*>(&st.gc[c0]) = gc;

            // decay factors and operand tiles
            // the early slot of this parity: both A-product warps are done with chunk c - 2
            if (g >= kEarly)
                ok = mbar_wait(&S.e_free[g & 1], (unsigned)(((g - kEarly) >> 1) & 1), err);
            if (!__all_sync(0xffffffffu, ok)) return false;
            unsigned char* x = reinterpret_cast<unsigned char*>(st.x);
            unsigned char* kge = reinterpret_cast<unsigned char*>(S.early[g & 1].kg);
            unsigned char* ki = reinterpret_cast<unsigned char*>(S.early[g & 1].ki);
            float kd0[4], kd1[4];
            __half v0[4], v1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + i;
                const float2 e = make_float2(ex2_approx(G[i].x), ex2_approx(G[i].y));
                const float2 d = make_float2(ex2_approx(-G[i].x), ex2_approx(-G[i].y));
                const float2 kv = bf2_to_f2(rk[i]);
                const float2 kg = f2mul(kv, e);
                const float2 kin = f2mul(kv, d);
                const float2 qg = f2mul(bf2_to_f2(rq[i]), e);
                const float2 kd = f2mul(kin, gc);
                const float2 vv = bf2_to_f2(rv[i]);
                *reinterpret_cast<float2*>(kge + tc::swizzled32_offset(r, c0, kChunk)) =
                    make_float2(tf32_round(kg.x), tf32_round(kg.y));
                *reinterpret_cast<float2*>(x + tc::swizzled32_offset(r, c0, X_ROWS)) =
                    make_float2(tf32_round(qg.x), tf32_round(qg.y));
                *reinterpret_cast<float2*>(ki + tc::swizzled32_offset(r, c0, kChunk)) =
                    make_float2(tf32_round(kin.x), tf32_round(kin.y));
                *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(st.kgh) + kgh_offset(r, c0)) =
                    pack_half2(kg.x, kg.y);
                kd0[i] = tf32_round(kd.x);
                kd1[i] = tf32_round(kd.y);
                v0[i] = __float2half_rn(vv.x);
                v1[i] = __float2half_rn(vv.y);
            }
            // (K 2^(G_last-G))^T and V^T: four consecutive tokens of one channel are
            // contiguous in the K-major core matrix
            unsigned char* kdt = reinterpret_cast<unsigned char*>(st.kdt);
            unsigned char* vt = reinterpret_cast<unsigned char*>(st.vt);
            *reinterpret_cast<float4*>(kdt + tc::interleaved32_offset(c0, r0, KD_SBO)) =
                make_float4(kd0[0], kd0[1], kd0[2], kd0[3]);
            *reinterpret_cast<float4*>(kdt + tc::interleaved32_offset(c0 + 1, r0, KD_SBO)) =
                make_float4(kd1[0], kd1[1], kd1[2], kd1[3]);
            *reinterpret_cast<uint2*>(vt + tc::interleaved16_offset(c0, r0, T_SBO)) =
                make_uint2(pack_halves(v0[0], v0[1]), pack_halves(v0[2], v0[3]));
            *reinterpret_cast<uint2*>(vt + tc::interleaved16_offset(c0 + 1, r0, T_SBO)) =
                make_uint2(pack_halves(v1[0], v1[1]), pack_halves(v1[2], v1[3]));
            // generic-proxy writes of this thread -> visible to the tensor core
            tc::fence_proxy_async_smem();
            mbar_arrive(&S.kq_ready[slot]);
        }
    }
    return true;
}

template <bool kP>
__device__ void produce(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S, int w, int lane,
                        int* err) {
    if constexpr (!kP) {
        produce_unit(P, U0, S, w, lane, err, 0);
    } else {
        int g = 0;
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, true, U)) return;
            if (!produce_unit(P, U, S, w, lane, err, g)) return;
            g += U.nch;
        }
    }
}

// ---- decay-ratio products (A-product warps) ----------------------------------------
// Warp 0 computes A_kk = (K 2^G)(K 2^-G)^T, warp 1 A_qk = (Q 2^G)(K 2^-G)^T, over the
// 128 key channels: m16n8k8 tf32 MMAs, fragments loaded with ldmatrix from the
// swizzled operand tiles (an 8 x 8 b16 matrix = 8 rows x 4 fp32).  Four independent
// accumulators per warp (two n-tiles x two channel halves) keep the MMA chains short;
// the halves are added in a fixed order.
__device__ __forceinline__ bool aprod_unit(const Unit& U, Smem& S, int which, int lane, int* err,
                                           int g0) {
    ProdShared& PS = S.pr;
    const int g = lane >> 2, t = lane & 3;
    const int m = lane >> 3, i8 = lane & 7;   // ldmatrix: matrix and row this lane addresses

    for (int c = 0; c < U.nch; ++c) {
        const int ck = g0 + c;   // chunk of the CTA
        const int par = ck & 1, slot = ck % kRing;
        bool ok = mbar_wait(&S.kq_ready[slot], (unsigned)((ck / kRing) & 1), err);
        // A_kk buffer of this parity: the solver is done with the chunk two before
        if (which == 0 && ck >= 2)
            ok = ok && mbar_wait(&S.t_ready[(ck - 2) % kRing], (unsigned)(((ck - 2) / kRing) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return false;
        Stage& st = S.st[slot];
        // A operand: K 2^G (early slot) or Q 2^G (rows 0-15 of the x tile)
        const unsigned char* xa = which ? reinterpret_cast<const unsigned char*>(st.x)
                                        : reinterpret_cast<const unsigned char*>(S.early[par].kg);
        const int xrows = which ? X_ROWS : kChunk;
        const unsigned char* ki = reinterpret_cast<const unsigned char*>(S.early[par].ki);
        float acc[2][2][4] = {};   // [channel half][n-tile][fragment]
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int k8 = kk + 8 * hh;
                // A: matrices (rows 0-7 | 8-15) x (channels 8 k8 .. +3 | +4 .. +7)
                // B: matrices (tokens 0-7 | 8-15) x (channels 8 k8 .. +3 | +4 .. +7)
                uint32_t a4[4], b4[4];
                ldsm_x4(a4, xa + tc::swizzled32_offset((m & 1) * 8 + i8, 8 * k8 + 4 * (m >> 1), xrows));
                ldsm_x4(b4, ki + tc::swizzled32_offset((m >> 1) * 8 + i8, 8 * k8 + 4 * (m & 1), kChunk));
                mma_tf32(acc[hh][0], a4, b4[0], b4[1]);
                mma_tf32(acc[hh][1], a4, b4[2], b4[3]);
            }
        }
        mbar_arrive(&S.e_free[par]);   // the early slot's tiles are no longer read
        // rows g, g + 8; columns (tokens s) 8 nt + 2t, + 1
        unsigned char* aqk = reinterpret_cast<unsigned char*>(st.aqk);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int s0 = 8 * nt + 2 * t;
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) r[e] = acc[0][nt][e] + acc[1][nt][e];
            if (which == 0) {
                *reinterpret_cast<float2*>(&PS.Akk[par][g * AK_LD + s0]) = make_float2(r[0], r[1]);
                *reinterpret_cast<float2*>(&PS.Akk[par][(g + 8) * AK_LD + s0]) = make_float2(r[2], r[3]);
            } else {   // A_qk inclusive lower (s <= row), tf32, K-major operand tile
                *reinterpret_cast<float2*>(aqk + tc::interleaved32_offset(g, s0, AQ_SBO)) =
                    make_float2(s0 <= g ? tf32_round(r[0]) : 0.0f, s0 + 1 <= g ? tf32_round(r[1]) : 0.0f);
                *reinterpret_cast<float2*>(aqk + tc::interleaved32_offset(g + 8, s0, AQ_SBO)) =
                    make_float2(s0 <= g + 8 ? tf32_round(r[2]) : 0.0f,
                                s0 + 1 <= g + 8 ? tf32_round(r[3]) : 0.0f);
            }
        }
        if (which == 1) {   // the A_qk tile is one of the chain's operands
            tc::fence_proxy_async_smem();
            mbar_arrive(&S.full[slot]);
        } else {
            mbar_arrive(&S.a_ready[par]);
        }
    }
    return true;
}

template <bool kP>
__device__ void aprod(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S, int which, int lane,
                      int* err) {
    if constexpr (!kP) {
        aprod_unit(U0, S, which, lane, err, 0);
    } else {
        int g = 0;
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, true, U)) return;
            if (!aprod_unit(U, S, which, lane, err, g)) return;
            g += U.nch;
        }
    }
}

// ---- w warps: -w = -T diag(b)(K 2^G) for channels 64 which .. + 63 -------------------
// fp16 m16n8k16 MMAs: A = T diag(b) (row-major fp16), B = K 2^G (fp16 [token][channel]);
// the result, negated and rounded to tf32, fills rows 16-31 of the x tile.
__device__ __forceinline__ bool wcalc_unit(const Unit& U, Smem& S, int which, int lane, int* err,
                                           int g0) {
    const int g = lane >> 2, t = lane & 3;
    for (int c = 0; c < U.nch; ++c) {
        const int ck = g0 + c;   // chunk of the CTA
        const int slot = ck % kRing;
        const bool ok = mbar_wait(&S.t_ready[slot], (unsigned)((ck / kRing) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return false;
        Stage& st = S.st[slot];
        unsigned char* x = reinterpret_cast<unsigned char*>(st.x);
        uint32_t ta[4];
        ldsm_x4(ta, &st.tbr[((lane & 7) + 8 * ((lane >> 3) & 1)) * TB_LD + 8 * (lane >> 4)]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // 16 channels per step: two n-tiles
            const int cb = 64 * which + 16 * q;
            uint32_t b[4];
            ldsm_x4_t(b, reinterpret_cast<const unsigned char*>(st.kgh) +
                             kgh_offset((lane & 7) + 8 * ((lane >> 3) & 1), cb + 8 * (lane >> 4)));
            float cw0[4] = {}, cw1[4] = {};
            mma_f16(cw0, ta, b[0], b[1]);
            mma_f16(cw1, ta, b[2], b[3]);
            const int col0 = cb + 2 * t, col1 = col0 + 8;
            *reinterpret_cast<float2*>(x + tc::swizzled32_offset(16 + g, col0, X_ROWS)) =
                make_float2(tf32_round(-cw0[0]), tf32_round(-cw0[1]));
            *reinterpret_cast<float2*>(x + tc::swizzled32_offset(24 + g, col0, X_ROWS)) =
                make_float2(tf32_round(-cw0[2]), tf32_round(-cw0[3]));
            *reinterpret_cast<float2*>(x + tc::swizzled32_offset(16 + g, col1, X_ROWS)) =
                make_float2(tf32_round(-cw1[0]), tf32_round(-cw1[1]));
            *reinterpret_cast<float2*>(x + tc::swizzled32_offset(24 + g, col1, X_ROWS)) =
                make_float2(tf32_round(-cw1[2]), tf32_round(-cw1[3]));
        }
        tc::fence_proxy_async_smem();   // -w is read by the chain's MMA
        mbar_arrive(&S.full[slot]);
    }
    return true;
}

template <bool kP>
__device__ void wcalc(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S, int which, int lane,
                      int* err) {
    if constexpr (!kP) {
        wcalc_unit(U0, S, which, lane, err, 0);
    } else {
        int g = 0;
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, true, U)) return;
            if (!wcalc_unit(U, S, which, lane, err, g)) return;
            g += U.nch;
        }
    }
}

// ---- solver warp: (I + diag(b) A_kk)^-1 and T diag(b) for every chunk -----------------
// A = diag(b) A_kk is strictly lower triangular, so A^16 = 0 and T = (I + A)^-1 is
// unit lower triangular.  Two evaluations, chosen per chunk:
//  - rho = max_i sum_m |A[i][m]| <= 1 (the usual case): the fp16 product
//      T = (I - A)(I + A^2)(I + A^4)(I + A^8)
//    ("Moonshot AI Open-Sources FlashKDA", "What makes the kernel fast": the 16 x 16
//    inverse in fp16), twelve m16n8k16 MMAs in registers; every power of A then has
//    entries of at most 1, so fp16 holds them;
//  - otherwise (keys of the chunk nearly parallel, b near 1, weak decay: the powers of
//    A grow to C(14, 7) = 3,432 while T stays small, and fp16 would lose the
//    cancellation) forward substitution in fp32,
//      T[i][:] = e_i - b_i sum_{m < i} A_kk[i][m] T[m][:],
//    lane j (and j + 16) forming column j, which keeps every intermediate the size of T.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}
// C fragments of a 16 x 16 product (two n-tiles) -> its A fragment and B fragments
__device__ __forceinline__ void frag_a(const float (&c)[2][4], uint32_t (&a)[4]) {
    a[0] = pack_half2(c[0][0], c[0][1]);
    a[1] = pack_half2(c[0][2], c[0][3]);
    a[2] = pack_half2(c[1][0], c[1][1]);
    a[3] = pack_half2(c[1][2], c[1][3]);
}
__device__ __forceinline__ void frag_b(const uint32_t (&a)[4], uint32_t (&b)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = movmatrix_t(a[i]);
}
// d = c + a * B (two n-tiles of 8 columns)
__device__ __forceinline__ void mma16(float (&d)[2][4], const uint32_t (&a)[4], const uint32_t (&b)[4]) {
    mma_f16(d[0], a, b[0], b[1]);
    mma_f16(d[1], a, b[2], b[3]);
}


// forward substitution of one chunk (the rare path, kept out of the solver's loop body)
__device__ __noinline__ void solve_substitution(const float* akk, float bl, int lane, __half* tbr,
                                                unsigned char* tbt) {
    const int j = lane & 15;   // column of T formed by this lane
    float tcol[kChunk];        // T[i][j]
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
        float acc0 = 0.0f, acc1 = 0.0f;   // two chains over m, added in a fixed order
#pragma unroll
        for (int q = 0; q < kChunk / 4; ++q) {
            if (4 * q < i) {
                const float4 a4 = *reinterpret_cast<const float4*>(akk + i * AK_LD + 4 * q);
                const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * q + e;
                    if (m < i) {
                        if (e & 1) acc1 = fmaf(a[e], tcol[m], acc1);
                        else acc0 = fmaf(a[e], tcol[m], acc0);
                    }
                }
            }
        }
        const float bi = __shfl_sync(0xffffffffu, bl, i);
        tcol[i] = (i == j ? 1.0f : 0.0f) - bi * (acc0 + acc1);
    }
    // T diag(b): column j scaled by b_j; lanes 0-15 write it row-major (A of w),
    // lanes 16-31 K-major (B of the u MMA)
    const float bj = __shfl_sync(0xffffffffu, bl, j);
    if (lane < 16) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) tbr[i * TB_LD + j] = __float2half_rn(tcol[i] * bj);
    } else {
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            *reinterpret_cast<__half*>(tbt + tc::interleaved_offset(i, j, kChunk)) =
                __float2half_rn(tcol[i] * bj);
    }
}

__device__ __forceinline__ bool solve_unit(const Problem& P, const Unit& U, Smem& S, int lane, int* err,
                                           int g0) {
    ProdShared& PS = S.pr;
    const int g = lane >> 2, t = lane & 3;
    // beta logits in windows of 64 tokens (4 chunks), the next window loaded one
    // window ahead: lane i holds tokens 64 j + i and 64 j + 32 + i of window j
    const __nv_bfloat16* beta = P.beta + (size_t)U.tok_start * P.H + U.h;
    const auto load_window = [&](int jw, float& w0, float& w1) {
        const int t0 = 64 * jw + lane, t1 = t0 + 32;
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
        // b of row `lane & 15`; rows past the sequence end get b = 0 (their T row is e_i)
        const float bl = ((lane & 15) < len) ? sigmoid_fast(lw) : 0.0f;
        const int ck = g0 + c;   // chunk of the CTA
        const int par = ck & 1;
        const bool ok = mbar_wait(&S.a_ready[par], (unsigned)((ck >> 1) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return false;
        Stage& st = S.st[ck % kRing];
        const float* akk = PS.Akk[par];
        unsigned char* tbt = reinterpret_cast<unsigned char*>(st.tbt);
        // A = diag(b) A_kk strictly lower, in accumulator layout (rows g, g + 8; columns
        // 8 nt + 2t, + 1), rounded to fp16; I - A; and the row sums of |A|
        const float bg = __shfl_sync(0xffffffffu, bl, g), bg8 = __shfl_sync(0xffffffffu, bl, g + 8);
        float cA[2][4], cI[2][4];
        float rs_g = 0.0f, rs_g8 = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float2 lo = *reinterpret_cast<const float2*>(&akk[g * AK_LD + 8 * nt + 2 * t]);
            const float2 hi = *reinterpret_cast<const float2*>(&akk[(g + 8) * AK_LD + 8 * nt + 2 * t]);
            const float raw[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = (e < 2) ? g : g + 8, col = 8 * nt + 2 * t + (e & 1);
                const float av =
                    (col < r) ? __half2float(__float2half_rn((e < 2 ? bg : bg8) * raw[e])) : 0.0f;
                cA[nt][e] = av;
                cI[nt][e] = (col == r ? 1.0f : 0.0f) - av;
                if (e < 2) rs_g += fabsf(av);
                else rs_g8 += fabsf(av);
            }
        }
        // rho = largest row sum: add over the four lanes of a row, then the maximum over
        // the warp (non-negative floats order like their bit patterns)
        rs_g += __shfl_xor_sync(0xffffffffu, rs_g, 1);
        rs_g8 += __shfl_xor_sync(0xffffffffu, rs_g8, 1);
        rs_g += __shfl_xor_sync(0xffffffffu, rs_g, 2);
        rs_g8 += __shfl_xor_sync(0xffffffffu, rs_g8, 2);
        const float rho =
            __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(rs_g, rs_g8))));
        if (rho <= 1.0f) {
            uint32_t aA[4], bA[4], aIA[4];
            frag_a(cA, aA);
            frag_b(aA, bA);
            frag_a(cI, aIA);
            float c2[2][4] = {}, c4[2][4] = {}, c8[2][4] = {};
            uint32_t aP[4], bA2[4], bA4[4], bA8[4];
            mma16(c2, aA, bA);                 // A^2
            frag_a(c2, aP);
            frag_b(aP, bA2);
            mma16(c4, aP, bA2);                // A^4
            mma16(cI, aIA, bA2);               // T1 = (I - A)(I + A^2)
            frag_a(c4, aP);
            frag_b(aP, bA4);
            mma16(c8, aP, bA4);                // A^8
            frag_a(cI, aP);
            mma16(cI, aP, bA4);                // T2 = T1 (I + A^4)
            frag_a(c8, aP);
            frag_b(aP, bA8);
            frag_a(cI, aP);
            mma16(cI, aP, bA8);                // T = T2 (I + A^8)
            // T diag(b): column n scaled by b_n; rows g, g+8, columns 8 nt + 2t, +1
            const float b0 = __shfl_sync(0xffffffffu, bl, 2 * t), b1 = __shfl_sync(0xffffffffu, bl, 2 * t + 1);
            const float b8 = __shfl_sync(0xffffffffu, bl, 8 + 2 * t), b9 = __shfl_sync(0xffffffffu, bl, 9 + 2 * t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float s0 = nt ? b8 : b0, s1 = nt ? b9 : b1;
                const uint32_t lo = pack_half2(cI[nt][0] * s0, cI[nt][1] * s1);   // row g
                const uint32_t hi = pack_half2(cI[nt][2] * s0, cI[nt][3] * s1);   // row g + 8
                const int col = 8 * nt + 2 * t;
                *reinterpret_cast<uint32_t*>(&st.tbr[g * TB_LD + col]) = lo;
                *reinterpret_cast<uint32_t*>(&st.tbr[(g + 8) * TB_LD + col]) = hi;
                *reinterpret_cast<uint32_t*>(tbt + tc::interleaved_offset(g, col, kChunk)) = lo;
                *reinterpret_cast<uint32_t*>(tbt + tc::interleaved_offset(g + 8, col, kChunk)) = hi;
            }
        } else {
            solve_substitution(akk, bl, lane, st.tbr, tbt);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive(&S.t_ready[ck % kRing]);
    }
    return true;
}

template <bool kP>
__device__ void solve(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S, int lane, int* err) {
    if constexpr (!kP) {
        solve_unit(P, U0, S, lane, err, 0);
    } else {
        int g = 0;
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, true, U)) return;
            if (!solve_unit(P, U, S, lane, err, g)) return;
            g += U.nch;
        }
    }
}

// ---- sequential stage: tensor-core issue (one thread) -------------------------------
// Per chunk c (slot s), in the transposed orientation (TMEM lane = value row v), with
// S^T of the chunk's start in state buffer c & 1:
//   [O|U] = S^T [Q 2^G ; -w]^T               (16 tf32 MMAs over the 128 key channels)
//   U    += V^T (T diag b)^T                  (u^T, fp16, after them)
//   S'^T += U^T (K 2^(G_last-G))              (S'^T = S^T 2^G_last, written by the
//                                              epilogue into the other state buffer)
//   O    += U^T A_qk^T
// The state and U are read from tensor memory as fp32 A operands (kind::tf32).
// One unit's chunks; g0 as for the loader, ui = this CTA's units with tokens before it.
// kZ: every unit starts from a zero state (no initial state given), so the first
// chunk's [O|U] MMAs would add exact zeros: they are left out, and u, the first O
// product and the first state update start fresh accumulators instead (the results
// are bit for bit those of a zero initial state).
// Returns the chunks whose MMAs and commits were all issued (fewer if a wait gave up).
template <bool kZ>
__device__ __forceinline__ int mma_unit(const Unit& U, Smem& S, uint32_t tmem, int* err, int g0,
                                        int ui) {
    constexpr uint32_t id_u = tc::idesc_f16_f32(128, 16);
    constexpr uint32_t id_s = tc::idesc_tf32_f32(128, 32);
    constexpr uint32_t id_k = tc::idesc_tf32_f32(128, 128);
    constexpr uint32_t id_q = tc::idesc_tf32_f32(128, 16);
    // descriptors of slot 0; slot s adds its byte offset >> 4 to the start field
    const uint64_t d_vt = tc::smem_desc(smem_u32(S.st[0].vt), 128, T_SBO, tc::kSwizzleNone);
    const uint64_t d_tbt = tc::smem_desc(smem_u32(S.st[0].tbt), 128, 256, tc::kSwizzleNone);
    const uint64_t d_xb = tc::smem_desc(smem_u32(S.st[0].x), 16, 1024, tc::kSwizzle128B);
    const uint64_t d_kdt = tc::smem_desc(smem_u32(S.st[0].kdt), 128, KD_SBO, tc::kSwizzleNone);
    const uint64_t d_aqk = tc::smem_desc(smem_u32(S.st[0].aqk), 128, AQ_SBO, tc::kSwizzleNone);
    int c = 0;
    for (; c < U.nch; ++c) {
        const int g = g0 + c;   // chunk of the CTA (the state and [O|U] buffers go by c)
        const int slot = g % kRing;
        const uint64_t so = (uint64_t)((slot * sizeof(Stage)) >> 4);
        const uint32_t sc = tmem + TM_S + 128u * (c & 1);
        const uint32_t sn = tmem + TM_S + 128u * ((c + 1) & 1);
        const uint32_t uo = tmem + TM_UO + 32u * (c % 3);
        if (!mbar_wait(&S.full[slot], (unsigned)((g / kRing) & 1), err)) break;
        if (c == 0) {
            if (!mbar_wait(&S.init_ready, (unsigned)(ui & 1), err)) break;
        } else {
            if (!mbar_wait(&S.s_done, (unsigned)((g - 1) & 1), err)) break;
        }
        tc::fence_after_sync();
        // with a zero state (kZ, first chunk) the products below that read it vanish
        uint32_t acc = 1;
        if constexpr (kZ) acc = c == 0 ? 0u : 1u;
        // [O|U] = S^T [Q 2^G ; -w]^T over the 16 key-channel steps (the first one starts
        // a fresh accumulator), then U += u^T = V^T (T diag b)^T
        if (acc) {
            tc::mma_ts_tf32(uo, sc, d_xb + so, id_s, 0);
#pragma unroll
            for (int kk = 1; kk < 16; ++kk)
                tc::mma_ts_tf32(uo, sc + 8 * kk,
                                d_xb + so + (uint64_t)(((kk >> 2) * X_ROWS * 128 + (kk & 3) * 32) >> 4),
                                id_s, 1);
        }
        tc::mma_ss(uo + 16, d_vt + so, d_tbt + so, id_u, acc);
        // one wait for both the [O|U] MMAs and the epilogue's rescale: a wait costs
        // this thread ~100 cycles even on a completed barrier
        tc::commit(smem_u32(&S.scaled));
        if (!mbar_wait(&S.scaled, (unsigned)(g & 1), err)) {
            // the [O|U] MMAs of this chunk were issued and committed: drain them below
            break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t a = kk == 0 ? acc : 1u;
            tc::mma_ts_tf32(sn, uo + 16 + 8 * kk, d_kdt + so + (uint64_t)((kk * 256) >> 4), id_k, a);
            tc::mma_ts_tf32(uo, uo + 16 + 8 * kk, d_aqk + so + (uint64_t)((kk * 256) >> 4), id_q, a);
        }
        tc::commit(smem_u32(&S.s_done));
        tc::commit(smem_u32(&S.empty[slot]));
    }
    return c;
}

template <bool kP, bool kZ>
__device__ void mma_issuer(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S,
                           uint32_t tmem, int* err) {
    int c = 0;   // chunks of this CTA whose commits were all issued
    if constexpr (!kP) {
        c = mma_unit<kZ>(U0, S, tmem, err, 0, 0);
    } else {
        int ui = 0;
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, false, U)) break;
            const int done = mma_unit<kZ>(U, S, tmem, err, c, ui);
            c += done;
            if (done < U.nch) break;   // a wait gave up
            if (U.nch > 0) ++ui;
        }
    }
    // Every MMA this thread issued completes before the CTA goes on to release tensor
    // memory and exit, also after a wait gave up part-way through a chunk: one more
    // commit, on a barrier of its own, tracks all of them.  Then the empty-slot commits
    // of the last chunks, which nobody else waits for, must have arrived: a late arrival
    // would hit the barrier that the next CTA on this SM initialises at the same
    // shared-memory address.
    tc::commit(smem_u32(&S.drain));
    mbar_wait(&S.drain, 0u, err, KDA_DRAIN_LIMIT);
    const int first = c > kRing ? c - kRing : 0;   // chunks 0 .. c - 1 were committed
    for (int i = first; i < c; ++i)
        mbar_wait(&S.empty[i % kRing], (unsigned)((i / kRing) & 1), err, KDA_DRAIN_LIMIT);
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
// Warp ew reaches TMEM lanes 32 ew .. + 31 (thread = value channel v) and owns all
// 128 state columns and the 16 outputs of those lanes.  Once the state of chunk c's
// start is complete, it writes 2^G_last(c) times it into the other state buffer,
// which the update MMAs of chunk c accumulate into while the U|O MMAs still read
// the first.
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

// One unit; g0 as for the loader.  kZ: zero initial state (nothing to write or rescale
// for the first chunk).  pre: this unit's first-chunk arrivals (init_ready, scaled) were
// made at the end of the unit before; post: make the next unit's at the end of this one,
// right after the last tensor-memory read and before the output stores (persistent CTAs
// with kZ, where those arrivals wait for nothing else).  Returns false if a wait gave up.
template <bool kZ>
__device__ __forceinline__ bool epilogue_unit(const Problem& P, const Unit& U, Smem& S,
                                              uint32_t tmem, int ew, int lane, int* err, int g0,
                                              bool pre = false, bool post = false) {
    const int v = 32 * ew + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * ew) << 16);   // this warp's lane quarter
    const size_t sbase = ((size_t)U.n * P.H + U.h) * kDim * kDim + v;   // + c * kDim
    bool ok = true;

    if (U.nch == 0) {   // no tokens: the final state is the initial state
        if (P.final_state)
            for (int c = 0; c < kDim; ++c)
                state_out(P, sbase + (size_t)c * kDim,
                          P.init_state ? state_in(P, sbase + (size_t)c * kDim) : 0.0f);
        return true;
    }
    // initial state S0 into buffer 0, then S0 Diag(2^G_last of chunk 0) into buffer 1
    if constexpr (!kZ) {
#pragma unroll 1
        for (int piece = 0; piece < 4; ++piece) {
            uint32_t x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 32 * piece + i;
                x[i] = __float_as_uint(P.init_state ? state_in(P, sbase + (size_t)c * kDim) : 0.0f);
            }
            tc::st32(tl + TM_S + 32 * piece, x);
        }
        tc::wait_st();
    }
    if (!pre) {
        tc::fence_before_sync();
        mbar_arrive(&S.init_ready);
        ok = mbar_wait(&S.full[g0 % kRing], (unsigned)((g0 / kRing) & 1), err);
        if (!__all_sync(0xffffffffu, ok)) return false;
    }
    if constexpr (!kZ) {
#pragma unroll 1
        for (int piece = 0; piece < 4; ++piece) {
            uint32_t x[32];
            tc::ld32(tl + TM_S + 32 * piece, x);
            tc::wait_ld();
            scale32(x, S.st[g0 % kRing].gc + 32 * piece);
            tc::st32(tl + TM_S + 128 + 32 * piece, x);
        }
        tc::wait_st();
    }
    if (!pre) {
        tc::fence_before_sync();
        mbar_arrive(&S.scaled);
    }

    // slot / phase of chunk c in the operand ring, and the [O|U] buffer of chunk c - 1
    int slot = (g0 + 1) % kRing, phase = ((g0 + 1) / kRing) & 1, uob = 0;
    __nv_bfloat16* out = P.out + ((size_t)U.tok_start * P.H + U.h) * kDim + v;
    const size_t out_step = (size_t)P.H * kDim;   // elements between consecutive tokens
    for (int c = 1; c <= U.nch; ++c) {
        // chunk c - 1 finished: its end state is in buffer c & 1
        ok = mbar_wait(&S.s_done, (unsigned)((g0 + c - 1) & 1), err);
        const bool more = c < U.nch;
        if (more) ok = ok && mbar_wait(&S.full[slot], (unsigned)phase, err);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc::fence_after_sync();
        const uint32_t sc = tl + TM_S + 128u * (c & 1);
        if (more) {
            const uint32_t sn = tl + TM_S + 128u * ((c + 1) & 1);
            const float* gc = S.st[slot].gc;
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t x[32];
                tc::ld32(sc + 32 * piece, x);
                tc::wait_ld();
                scale32(x, gc + 32 * piece);
                tc::st32(sn + 32 * piece, x);
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(&S.scaled);
        } else if (P.final_state) {
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t x[32];
                tc::ld32(sc + 32 * piece, x);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    state_out(P, sbase + (size_t)(32 * piece + i) * kDim, __uint_as_float(x[i]));
            }
        }
        // outputs of chunk c - 1: O^T lane v, column t = token
        {
            uint32_t o[16];
            tc::ld16(tl + TM_UO + 32u * uob, o);
            tc::wait_ld();
            if (post && !more) {   // tensor memory read for the last time: the next unit may start
                tc::fence_before_sync();
                mbar_arrive(&S.init_ready);
                mbar_arrive(&S.scaled);
            }
            const int len = min(kChunk, U.L - (c - 1) * kChunk);
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
                if (t < len) out[t * out_step] = __float2bfloat16_rn(P.scale * __uint_as_float(o[t]));
            out += kChunk * out_step;
        }
        if (++slot == kRing) {
            slot = 0;
            phase ^= 1;
        }
        if (++uob == 3) uob = 0;
    }
    return true;
}

template <bool kP, bool kZ>
__device__ void epilogue(const Problem& P, const SeqMap& M, const Unit& U0, Smem& S, uint32_t tmem,
                         int ew, int lane, int* err) {
    if constexpr (!kP) {
        epilogue_unit<kZ>(P, U0, S, tmem, ew, lane, err, 0);
    } else {
        int g = 0;
        bool pre = false;   // the arrivals of the next unit with tokens were made early
        for (int k = 0;; ++k) {
            Unit U;
            if (!read_unit(S, k, err, true, U)) return;
            if (!epilogue_unit<kZ>(P, U, S, tmem, ew, lane, err, g, pre, kZ)) return;
            if (U.nch > 0) pre = kZ;   // a unit without tokens makes and takes no arrivals
            g += U.nch;
        }
    }
}

// kP: persistent (a grid of at most one CTA per SM takes the units from a device
// counter, longest first); otherwise one CTA per unit.  Every unit's arithmetic is the
// same either way.  kZ: no initial state (every unit starts from zero).
template <bool kP, bool kZ>
__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(Problem P, SeqMap M, const __grid_constant__ RawMaps TM, int* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzle acts on absolute shared addresses: align the stages to 1024 B
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Smem& S = *reinterpret_cast<Smem*>(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    Unit U;
    if constexpr (kP) {
        if (!*M.valid) return;  // malformed cu_seqlens: write nothing (CTA-uniform)
        U = Unit{};
    } else {
        U.h = blockIdx.x % P.H;
        const int rank = blockIdx.x / P.H;
        U.vzero = false;
        if (P.window >= 0) {
            // sequence split (fixed length): the unit's sequence, segment and kind.  Its
            // initial state (prepared on the host side: the caller's, zero or identity) and
            // its final state are at index rank of fp32 scratch.
            const int per = P.window == 0 ? 2 * P.nseg - 3 : P.nseg - 1;
            const int seq = rank / per, vj = rank % per;
            int j = P.window == 0 ? vj : vj + 1;      // segment
            if (P.window == 0 && vj > P.nseg - 2) {
                j = vj - (P.nseg - 2);                // transition operator: zero values
                U.vzero = true;
            }
            U.n = rank;
            const long long nchk = (P.T + kChunk - 1) / kChunk;
            const int c0 = (int)((long long)j * nchk / P.nseg);
            const int c1 = (int)((long long)(j + 1) * nchk / P.nseg);
            U.tok_start = seq * P.T + c0 * kChunk;
            U.L = min(c1 * kChunk, P.T) - c0 * kChunk;
        } else if (P.cu_seqlens == nullptr) {
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
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&S.full[s], 96);             // both w warps and the A_qk warp
            mbar_init(&S.empty[s], 1);             // one tensor-core commit
            mbar_init(&S.kq_ready[s], kProdThreads);   // every producer thread
            mbar_init(&S.t_ready[s], 32);          // solver warp
        }
        for (int s = 0; s < kEarly; ++s) mbar_init(&S.e_free[s], 64);   // both A-product warps
        mbar_init(&S.s_done, 1);
        mbar_init(&S.init_ready, kEpiWarps * 32);
        mbar_init(&S.scaled, kEpiWarps * 32 + 1);   // epilogue threads + one commit
        mbar_init(&S.epi_done, kEpiWarps * 32);
        mbar_init(&S.drain, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.a_ready[b], 32);              // the A_kk warp
        }
        for (int s = 0; s < kRaw; ++s) {
            mbar_init(&S.raw_full[s], 1);                 // loader's arrive + TMA bytes
            mbar_init(&S.raw_empty[s], kProdThreads);     // every producer thread
        }
        if (kP) {
            for (int s = 0; s < kUnitRing; ++s) {
                mbar_init(&S.unit_full[s], 1);               // the loader
                mbar_init(&S.unit_empty[s], kUnitReaders);   // one arrival per reading warp
            }
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
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

    const Role role = role_of(warp);
    if (role == kEpi) {
        epilogue<kP, kZ>(P, M, U, S, tmem, warp, lane, err);
        tc::fence_before_sync();
        mbar_arrive(&S.epi_done);
    } else if (role == kMma) {
        if (lane == 0) mma_issuer<kP, kZ>(P, M, U, S, tmem, err);
        __syncwarp();
        // free tensor memory once the epilogue is done with it (after a timeout the
        // epilogue stops at its next wait, so a longer limit than a pipeline wait's)
        const bool ok = mbar_wait(&S.epi_done, 0u, err, KDA_DRAIN_LIMIT);
        __syncwarp();
        (void)ok;
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    } else if (role == kSolve) {
        solve<kP>(P, M, U, S, lane, err);
    } else if (role == kAprod0 || role == kAprod1) {
        aprod<kP>(P, M, U, S, role == kAprod1, lane, err);
    } else if (role == kW0 || role == kW1) {
        wcalc<kP>(P, M, U, S, role == kW1, lane, err);
    } else if (role == kLoad) {
        if (lane == 0) loader<kP>(P, M, TM, U, S, err);
    } else {
        produce<kP>(P, M, U, S, prod_index(warp), lane, err);
    }
}

// per-device flag: the kernel attribute below is set once (setting it is idempotent,
// so two threads racing on a first call both succeed)
std::atomic<bool> g_attr_set[64];
std::atomic<int> g_sms[64];   // SM count per device, 0 until read

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
    if (dev >= 0 && dev < 64 && !g_attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(fused_kernel<false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fused_kernel<true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fused_kernel<false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fused_kernel<true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sms[dev].store(sms, std::memory_order_relaxed);
        g_attr_set[dev].store(true, std::memory_order_release);
    }
    const long long per = P.window == 0 ? 2LL * P.nseg - 3 : P.window == 1 ? P.nseg - 1LL : 1LL;
    const long long ctas = (long long)P.N * P.H * per;
    if (ctas == 0) return cudaSuccess;
    // more varlen units than SMs, and a unit counter given: one persistent CTA per SM
    const int sms = (dev >= 0 && dev < 64) ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    const bool persist = P.cu_seqlens != nullptr && M.counter != nullptr && sms > 0 && ctas > sms;
    // total token rows: B*T (fixed length, N = B sequences of T) or T (varlen, B = 1)
    const long long rows = (P.cu_seqlens == nullptr) ? (long long)P.N * P.T : (long long)P.T;
    RawMaps TM;
    memset(&TM, 0, sizeof(TM));
    if (rows > 0) {
        cudaError_t e = encode_rows(&TM.q, P.q, P.H, rows);
        if (e == cudaSuccess) e = encode_rows(&TM.k, P.k, P.H, rows);
        if (e == cudaSuccess) e = encode_rows(&TM.v, P.v, P.H, rows);
        // 16 zero rows for the units with zero values (window 0 of a split call)
        if (e == cudaSuccess && P.vzero) e = encode_rows(&TM.vz, P.vzero, P.H, kChunk);
        if (e == cudaSuccess) e = encode_rows(&TM.g, P.g, P.H, rows);
        if (e != cudaSuccess) return e;
    }   // else no tokens: the loader issues nothing
    const bool zero = P.init_state == nullptr;   // every unit starts from a zero state
    if (persist && zero)
        fused_kernel<true, true><<<(unsigned)sms, kThreads, smem, s>>>(P, M, TM, err);
    else if (persist)
        fused_kernel<true, false><<<(unsigned)sms, kThreads, smem, s>>>(P, M, TM, err);
    else if (zero)
        fused_kernel<false, true><<<(unsigned)ctas, kThreads, smem, s>>>(P, M, TM, err);
    else
        fused_kernel<false, false><<<(unsigned)ctas, kThreads, smem, s>>>(P, M, TM, err);
    return cudaGetLastError();
}

}  // namespace kda
