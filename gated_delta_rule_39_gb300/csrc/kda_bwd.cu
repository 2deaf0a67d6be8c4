// KDA backward pass: the gradients of a loss with respect to q, k, v, g, beta, A_log,
// dt_bias and the initial state, given its gradients with respect to the outputs
// (and, optionally, the final state).  The pages' library is forward-only ("Moonshot
// AI Open-Sources FlashKDA", "Limitations before you integrate"); this is the reverse
// pass of the same recurrence (the forward's reading is in kda.h):
//
//   x_t = exp(A_log) (g_t + dt_bias),  a_t = exp(lower_bound sigmoid(x_t)),  b_t = sigmoid(beta_t)
//   S'_t = Diag(a_t) S_{t-1},  r_t = S'_t^T k_t,  d_t = b_t (v_t - r_t),  S_t = S'_t + k_t d_t^T
//   o_t = scale S_t^T q_t
//
// Reverse, carrying dS = dL/dS_t from the last token to the first:
//   dS += scale q dO^T;   dq = scale S_t dO;   dd = dS^T k;   dk = dS d;   dv = b dd;
//   db = dd . (v - r);   dr = -b dd;   dS' = dS + k dr^T;   dk += S' dr;
//   da = rowsum(dS' o S_{t-1});   dS = Diag(a) dS'
// and the activations' chain rule for dg, dt_bias, A_log and beta.
//
// The value columns of the state are independent recurrences (k, a and b are shared),
// so the work is cut into 8 slices of 16 value columns per (sequence, head), one CTA
// of 4 warps each.  Lane l of warp w holds S[4l .. 4l + 3][16 s + 4w .. 4w + 3]: a warp
// holds all 128 keys of 4 columns, so the sums over value columns (dq, dk, da) are
// sums in registers, and the sums over keys (r = S'^T k, dd = dS^T k, one per column)
// are one reduce-scatter and broadcast over the warp (10 shuffles for the 4 columns).
// Each block of 8 token rows is staged in shared memory at once, its raw rows loaded
// into registers one block ahead.  Phase 1 runs the slice forward, storing its state
// every 8 tokens and each token's d and v - r; phase 2 walks the blocks backwards,
// and each block's halves backwards: it rebuilds the half's states from the checkpoint
// (the same arithmetic as phase 1, element-wise, with the stored d) into shared memory
// and runs the reverse steps over them.
// The 4 warps' sums of dq, dk, da and db wait in shared memory and are added every 4
// tokens; the 8 slices' sums are added by a second kernel (every sum in a fixed
// order), which also applies the activations.  This is a token-by-token pass on CUDA
// cores; a chunked pass on tensor cores, as the forward is, would be much faster.
#include <atomic>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kSlices = 8;          // value slices per (sequence, head)
constexpr int kSliceV = kDim / kSlices;   // 16 value columns
constexpr int kBwdWarps = 4;        // 4 value columns each
constexpr int kBwdThreads = 32 * kBwdWarps;
constexpr int kPart = 388;          // partial sums per (row, head, slice): dq, dk, da [128], db
constexpr int kGroup = 4;           // tokens whose per-warp partial sums wait in shared memory
constexpr int kBC = 8;              // tokens per checkpoint (and per staged block of rows)
constexpr int kHalf = kBC / 2;      // states rebuilt at a time (half a block): with these
                                    // sizes three CTAs fit on an SM
constexpr int kCkFloats = kDim * kSliceV;   // one slice's state: 16 floats per thread

struct BwdSmem {
    float4 st[kHalf][4][kBwdThreads];   // S_{t-1} of each token of half a block: a thread's
                                        // 16 values as 4 float4 planes (one per column)
    float a[kBC][kDim];                  // the block's decays
    float kk[kBC][kDim];                 // keys
    float qq[kBC][kDim];                 // queries (reverse phase)
    float vv[kBC][kSliceV];             // the slice's values (forward) or dL/d(out) (reverse)
    float fw[kBC][2 * kSliceV];         // d and v - r of the slice (reverse)
    float b[kBC];                       // sigmoid(beta)
    // reverse: per-warp sums over the warp's 4 columns of dq, dk, da (128 keys each) and
    // db, for a group of tokens; summed over the 4 warps once per group
    float grp[kGroup][kBwdWarps][3 * kDim + 4];
};

__device__ __forceinline__ float bf(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }

// sigmoid and the decay from CUDA's fast exponential and reciprocal intrinsics (relative
// error ~1e-7, far inside the gradients' tolerance; every kernel of the pass uses these
// same two functions, so phase 1, phase 2 and the finish kernel see the same bits)
__device__ __forceinline__ float sigm(float x) { return __frcp_rn(1.0f + __expf(-x)); }
__device__ __forceinline__ float decay_of(float x, float lower_bound) {
    return __expf(lower_bound * sigm(x));
}

// the decay of key channel c at token row t, and x (the sigmoid's argument)
__device__ __forceinline__ float decay(const BwdProblem& P, size_t row, int h, int c, float eA,
                                      float* xo = nullptr) {
    const float x = eA * (bf(P.g, (row * P.H + h) * kDim + c) + P.dt_bias[(size_t)h * kDim + c]);
    if (xo) *xo = x;
    return decay_of(x, P.lower_bound);
}

// Checkpoint slot of block c (of 8 tokens) of sequence n (first token bos): distinct for
// every (n, c) of a call, below N + rows / 8 + 1.
__device__ __forceinline__ long long ck_slot(int n, long long bos, int c) {
    return (long long)n + c + bos / kBC;
}

// A block's raw token rows, loaded into registers one block ahead of their use, so that
// their memory latency overlaps the block before: keys, gate inputs (and queries on the
// way back) as thread (row, 8 channels); in x, the slice's 16 values or dL/d(out)
// (threads 0-15, 8 columns each), the beta logit (threads 16-23) or the stored d and
// v - r on the way back (threads 64-127, 4 floats each).  Rows past the sequence's end
// are not read.
struct Rows {
    uint4 k, g, q;
    uint4 x;
};

__device__ __forceinline__ void fetch(const BwdProblem& P, Rows& R, long long row0, int len,
                                      int h, int col0, bool reverse, const float* fw0,
                                      size_t fw_step) {
    const int tid = threadIdx.x;
    const int i = tid >> 4, c8 = 8 * (tid & 15);
    if (i < len) {
        const size_t rk = ((size_t)(row0 + i) * P.H + h) * kDim + c8;
        R.k = *reinterpret_cast<const uint4*>(P.k + rk);
        R.g = *reinterpret_cast<const uint4*>(P.g + rk);
        if (reverse) R.q = *reinterpret_cast<const uint4*>(P.q + rk);
    }
    if (tid < 2 * kBC) {
        const int r = tid >> 1, hv = tid & 1;
        if (r < len) {
            const size_t rv = ((size_t)(row0 + r) * P.H + h) * kDim + col0 + 8 * hv;
            R.x = *reinterpret_cast<const uint4*>(reverse ? P.dout + rv : P.v + rv);
        }
    } else if (tid < 3 * kBC) {
        const int r = tid - 2 * kBC;
        if (r < len) R.x.x = __float_as_uint(bf(P.beta, (size_t)(row0 + r) * P.H + h));
    } else if (reverse && tid >= 64 && tid < 64 + 8 * kBC) {
        const int r = (tid - 64) >> 3, f4 = 4 * ((tid - 64) & 7);
        if (r < len) R.x = *reinterpret_cast<const uint4*>(fw0 + (size_t)r * fw_step + f4);
    }
}

__device__ __forceinline__ void unpack8(uint4 w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[2 * j] = __uint_as_float(u[j] << 16);
        x[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void st8(float* p, const float (&x)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
}

// The fetched rows into shared memory (decays and b formed on the way), then a barrier.
// dtb: dt_bias of the thread's 8 channels.
__device__ __forceinline__ void commit(BwdSmem& S, const Rows& R, int len, float eA,
                                       float lower_bound, const float (&dtb)[8], bool reverse) {
    const int tid = threadIdx.x;
    const int i = tid >> 4, c8 = 8 * (tid & 15);
    if (i < len) {
        float kx[8], gx[8], a[8];
        unpack8(R.k, kx);
        unpack8(R.g, gx);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = decay_of(eA * (gx[e] + dtb[e]), lower_bound);
        st8(&S.a[i][c8], a);
        st8(&S.kk[i][c8], kx);
        if (reverse) {
            float qx[8];
            unpack8(R.q, qx);
            st8(&S.qq[i][c8], qx);
        }
    }
    if (tid < 2 * kBC) {
        const int r = tid >> 1, hv = tid & 1;
        if (r < len) {
            float x[8];
            unpack8(R.x, x);
            st8(&S.vv[r][8 * hv], x);
        }
    } else if (tid < 3 * kBC) {
        const int r = tid - 2 * kBC;
        if (r < len) S.b[r] = sigm(__uint_as_float(R.x.x));
    } else if (reverse && tid >= 64 && tid < 64 + 8 * kBC) {
        const int r = (tid - 64) >> 3, f4 = 4 * ((tid - 64) & 7);
        if (r < len)
            *reinterpret_cast<float4*>(&S.fw[r][f4]) =
                make_float4(__uint_as_float(R.x.x), __uint_as_float(R.x.y),
                            __uint_as_float(R.x.z), __uint_as_float(R.x.w));
    }
    __syncthreads();
}

// Packed fp32 pairs (one instruction for two lanes' worth of arithmetic), each with an
// explicit round-to-nearest so that no multiply and add are fused behind the code's
// back: phase 2 replays phase 1's state updates and must get the same bits.
__device__ __forceinline__ unsigned long long pk2(float2 a) {
    unsigned long long x;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    return x;
}
__device__ __forceinline__ float2 upk2(unsigned long long x) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long z;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(z);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long z;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(z);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long z;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(z) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return upk2(z);
}
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }

// The sums over the warp's 32 lanes of 4 per-column partial sums p[0..3], returned in
// every lane: lanes halve the columns they keep at xor 16 and xor 8 (after which lane l
// keeps column 2 (l >> 4 & 1) + (l >> 3 & 1)), sum that one over xor 4, 2, 1, and
// fetch the four results from lanes 0, 8, 16 and 24.  A fixed order: every lane gets
// the same bits.
__device__ __forceinline__ void warp_sum4(float (&p)[4], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8;
    float k0 = h16 ? p[2] : p[0], k1 = h16 ? p[3] : p[1];
    const float s0 = h16 ? p[0] : p[2], s1 = h16 ? p[1] : p[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    float k = h8 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
    k += __shfl_xor_sync(0xffffffffu, k, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    p[0] = __shfl_sync(0xffffffffu, k, 0);
    p[1] = __shfl_sync(0xffffffffu, k, 8);
    p[2] = __shfl_sync(0xffffffffu, k, 16);
    p[3] = __shfl_sync(0xffffffffu, k, 24);
}

__device__ __forceinline__ void ld_keys(const float* row, int lane, float2 (&x)[2]) {
    const float4 u = *reinterpret_cast<const float4*>(row + 4 * lane);
    x[0] = make_float2(u.x, u.y);
    x[1] = make_float2(u.z, u.w);
}

__device__ __forceinline__ float4 f4(const float2 (&x)[2]) {
    return make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
}

__global__ void __launch_bounds__(kBwdThreads, 3) bwd_kernel(BwdProblem P, const int* valid) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem& S = *reinterpret_cast<BwdSmem*>(smem_raw);
    if (valid && !*valid) return;   // malformed cu_seqlens: the sequence map says so
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x % kSlices;
    const int h = (blockIdx.x / kSlices) % P.H;
    const int n = blockIdx.x / (kSlices * P.H);
    const long long bos = P.cu_seqlens ? P.cu_seqlens[n] : (long long)n * P.T;
    const int L = P.cu_seqlens ? P.cu_seqlens[n + 1] - P.cu_seqlens[n] : P.T;
    const int nch = (L + kBC - 1) / kBC;
    const int col0 = kSliceV * slice;
    const int j0 = 4 * warp;               // the warp's first column within the slice
    const float eA = expf(P.A_log[h]);
    const size_t fw_step = (size_t)P.H * kSlices * (2 * kSliceV);           // between rows
    const auto fw_at = [&](size_t row) {   // d (16) and v - r (16) of this slice at a row
        return P.fw + ((row * P.H + h) * kSlices + slice) * (2 * kSliceV);
    };
    // checkpoint of block c: the slice's state, 16 floats per thread (4 float4, one per
    // column), written and read back by the same thread
    const auto ck_at = [&](int c) {
        return P.ck + ((ck_slot(n, bos, c) * P.H + h) * kSlices + slice) * kCkFloats + 16 * tid;
    };
    float dtb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) dtb[e] = P.dt_bias[(size_t)h * kDim + 8 * (tid & 15) + e];
    // element (key 4 lane + 2 p + x, column j0 + c) of the slice's state in [c][p].x|y
    const auto state_index = [&](int key, int c) {
        return (((size_t)n * P.H + h) * kDim + key) * kDim + col0 + j0 + c;
    };
    Rows R{};

    // ---- phase 1: forward over the slice, checkpoints and per-token d, v - r ----------
    {
        float2 st[4][2];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = 0.0f;
                if (P.init_state) {
                    const size_t si = state_index(4 * lane + e, c);
                    x = P.init_dtype == KDA_F32
                            ? static_cast<const float*>(P.init_state)[si]
                            : __bfloat162float(static_cast<const __nv_bfloat16*>(P.init_state)[si]);
                }
                if (e & 1) st[c][e >> 1].y = x; else st[c][e >> 1].x = x;
            }
        if (nch > 0) fetch(P, R, bos, min(kBC, L), h, col0, false, nullptr, 0);
        for (int c = 0; c < nch; ++c) {
            float4* ck = reinterpret_cast<float4*>(ck_at(c));
#pragma unroll
            for (int j = 0; j < 4; ++j) ck[j] = f4(st[j]);
            const int len = min(kBC, L - c * kBC);
            const long long row0 = bos + (long long)c * kBC;
            commit(S, R, len, eA, P.lower_bound, dtb, false);
            if (c + 1 < nch)
                fetch(P, R, row0 + kBC, min(kBC, L - (c + 1) * kBC), h, col0, false, nullptr, 0);
            for (int i = 0; i < len; ++i) {
                float2 a[2], kk[2];
                ld_keys(S.a[i], lane, a);
                ld_keys(S.kk[i], lane, kk);
                const float4 v4 = *reinterpret_cast<const float4*>(&S.vv[i][j0]);
                const float v[4] = {v4.x, v4.y, v4.z, v4.w};
                const float b = S.b[i];
                float r[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 rp = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        st[j][p] = mul2(st[j][p], a[p]);
                        rp = fma2(st[j][p], kk[p], rp);
                    }
                    r[j] = rp.x + rp.y;
                }
                warp_sum4(r, lane);
                float d[4], vr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    vr[j] = v[j] - r[j];
                    d[j] = b * vr[j];
#pragma unroll
                    for (int p = 0; p < 2; ++p) st[j][p] = fma2(kk[p], dup2(d[j]), st[j][p]);
                }
                if (lane == 0) {   // the warp's 4 columns of d and v - r
                    float* f = fw_at(row0 + i);
                    *reinterpret_cast<float4*>(f + j0) = make_float4(d[0], d[1], d[2], d[3]);
                    *reinterpret_cast<float4*>(f + kSliceV + j0) = make_float4(vr[0], vr[1], vr[2], vr[3]);
                }
            }
            __syncthreads();   // the staged rows are replaced by the next block's
        }
    }
    __syncthreads();   // d and v - r are read by other threads below

    // ---- phase 2: reverse, block by block from the last ---------------------------------
    float2 dS[4][2];
    float4 ckn[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x = P.dfinal ? P.dfinal[state_index(4 * lane + e, c)] : 0.0f;
            if (e & 1) dS[c][e >> 1].y = x; else dS[c][e >> 1].x = x;
        }
    if (nch > 0) {
        const long long row0 = bos + (long long)(nch - 1) * kBC;
        fetch(P, R, row0, L - (nch - 1) * kBC, h, col0, true, fw_at(row0), fw_step);
        const float4* ck = reinterpret_cast<const float4*>(ck_at(nch - 1));
#pragma unroll
        for (int j = 0; j < 4; ++j) ckn[j] = ck[j];   // written by this thread
    }
    for (int c = nch - 1; c >= 0; --c) {
        const int len = min(kBC, L - c * kBC);
        const long long row0 = bos + (long long)c * kBC;
        commit(S, R, len, eA, P.lower_bound, dtb, true);
        float2 sv[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sv[j][0] = make_float2(ckn[j].x, ckn[j].y);
            sv[j][1] = make_float2(ckn[j].z, ckn[j].w);
        }
        if (c > 0) {   // the block before is whole
            fetch(P, R, row0 - kBC, kBC, h, col0, true, fw_at(row0 - kBC), fw_step);
            const float4* ck = reinterpret_cast<const float4*>(ck_at(c - 1));
#pragma unroll
            for (int j = 0; j < 4; ++j) ckn[j] = ck[j];
        }
        // The block's two halves, the later first: rebuild the half's states S_{t-1} from
        // the checkpoint (the same arithmetic as phase 1, stepping over the first half
        // for the later one; each thread reads back only its own states), then run the
        // reverse steps over the half.
        for (int lo = len > kHalf ? kHalf : 0; lo >= 0; lo -= kHalf) {
            const int hi = min(len, lo + kHalf);
            float2 s2[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s2[j][0] = sv[j][0];
                s2[j][1] = sv[j][1];
            }
            for (int i = 0; i < hi; ++i) {
                float2 a[2], kk[2];
                ld_keys(S.a[i], lane, a);
                ld_keys(S.kk[i], lane, kk);
                const float4 d4 = *reinterpret_cast<const float4*>(&S.fw[i][j0]);
                const float d[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (i >= lo) S.st[i - lo][j][tid] = f4(s2[j]);
#pragma unroll
                    for (int p = 0; p < 2; ++p) s2[j][p] = fma2(kk[p], dup2(d[j]), mul2(s2[j][p], a[p]));
                }
            }
            for (int i = hi - 1; i >= lo; --i) {
                const int gi = (len - 1 - i) % kGroup;   // slot of this token in its group
                float2 a[2], kk[2], qq[2];
                ld_keys(S.a[i], lane, a);
                ld_keys(S.kk[i], lane, kk);
                ld_keys(S.qq[i], lane, qq);
                const float4 d4 = *reinterpret_cast<const float4*>(&S.fw[i][j0]);
                const float4 vr4 = *reinterpret_cast<const float4*>(&S.fw[i][kSliceV + j0]);
                const float4 do4 = *reinterpret_cast<const float4*>(&S.vv[i][j0]);
                const float d[4] = {d4.x, d4.y, d4.z, d4.w};
                const float vr[4] = {vr4.x, vr4.y, vr4.z, vr4.w};
                const float dout[4] = {do4.x, do4.y, do4.z, do4.w};
                const float b = S.b[i];
                float2 sprev[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 s4 = S.st[i - lo][j][tid];
                    sprev[j][0] = make_float2(s4.x, s4.y);
                    sprev[j][1] = make_float2(s4.z, s4.w);
                }
                const float2 zero = make_float2(0.0f, 0.0f);
                float2 dq[2] = {zero, zero}, dk[2] = {zero, zero}, da[2] = {zero, zero};
                float dd[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 ddp = zero;
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float2 sp = mul2(sprev[j][p], a[p]);
                        // S_t dO (scale applied when the warps' sums are added)
                        dq[p] = fma2(fma2(kk[p], dup2(d[j]), sp), dup2(dout[j]), dq[p]);
                        dS[j][p] = fma2(qq[p], dup2(P.scale * dout[j]), dS[j][p]);
                        dk[p] = fma2(dS[j][p], dup2(d[j]), dk[p]);
                        ddp = fma2(dS[j][p], kk[p], ddp);
                    }
                    dd[j] = ddp.x + ddp.y;
                }
                warp_sum4(dd, lane);   // dd = dS^T k over the 128 keys, per column
                float db = 0.0f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 dr = dup2(-b * dd[j]);
                    db = fmaf(dd[j], vr[j], db);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float2 sp = mul2(sprev[j][p], a[p]);
                        const float2 dsp = fma2(kk[p], dr, dS[j][p]);
                        dk[p] = fma2(sp, dr, dk[p]);
                        da[p] = fma2(dsp, sprev[j][p], da[p]);
                        dS[j][p] = mul2(a[p], dsp);
                    }
                }
                const size_t row = row0 + i;
                if (lane == 0) {
                    *reinterpret_cast<float4*>(P.dv + (row * P.H + h) * kDim + col0 + j0) =
                        make_float4(b * dd[0], b * dd[1], b * dd[2], b * dd[3]);
                    S.grp[gi][warp][3 * kDim] = db;
                }
                float* gp = S.grp[gi][warp];
                *reinterpret_cast<float4*>(gp + 4 * lane) = f4(dq);
                *reinterpret_cast<float4*>(gp + kDim + 4 * lane) = f4(dk);
                *reinterpret_cast<float4*>(gp + 2 * kDim + 4 * lane) = f4(da);
                if (gi == kGroup - 1 || i == 0) {
                    // the group's tokens (rows row .. row + gi): sum the 4 warps in order and
                    // write this slice's partial sums
                    __syncthreads();
                    if (tid < kPart / 4) {   // one float4 of each token's 388 sums per thread
                        const int e = 4 * tid;   // dq (scaled), dk, da; the last holds db
                        const float2 sc = dup2(e < kDim ? P.scale : 1.0f);
                        for (int g = 0; g <= gi; ++g) {
                            const size_t grow = row + gi - g;   // slot g: the g-th token walked
                            float2 lo = zero, hi = zero;
#pragma unroll
                            for (int w = 0; w < kBwdWarps; ++w) {
                                const float4 x = *reinterpret_cast<const float4*>(&S.grp[g][w][e]);
                                lo = add2(lo, make_float2(x.x, x.y));
                                hi = add2(hi, make_float2(x.z, x.w));
                            }
                            lo = mul2(lo, sc);
                            hi = mul2(hi, sc);
                            *reinterpret_cast<float4*>(P.part + ((grow * P.H + h) * kSlices + slice) * kPart + e) =
                                make_float4(lo.x, lo.y, hi.x, hi.y);
                        }
                    }
                    __syncthreads();
                }
            }
        }
        __syncthreads();   // the block's staged rows and states are replaced by the next one
    }
    if (P.d_init) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int p = e >> 1;
            const auto x = [&](int j) { return (e & 1) ? dS[j][p].y : dS[j][p].x; };
            *reinterpret_cast<float4*>(P.d_init + state_index(4 * lane + e, 0)) =
                make_float4(x(0), x(1), x(2), x(3));
        }
    }
}

// ---- finish: slices summed in a fixed order, activations' chain rule ------------------
// One CTA of 128 threads (thread = key channel) per (head, block of 64 token rows);
// writes dq, dk, dg, dbeta, and the block's sums of dg (for dt_bias) and of
// dx . x (for A_log).
constexpr int kRowBlock = 64;

__global__ void __launch_bounds__(kDim) bwd_finish_kernel(BwdProblem P, long long rows,
                                                          const int* valid) {
    __shared__ float red[kDim / 32];
    if (valid && !*valid) return;
    const int c = threadIdx.x;
    const int h = blockIdx.x % P.H;
    const long long blk = blockIdx.x / P.H;
    const float eA = expf(P.A_log[h]);
    float sdg = 0.0f, sdA = 0.0f;
    const long long r0 = blk * kRowBlock, r1 = min(rows, r0 + kRowBlock);
    for (long long row = r0; row < r1; ++row) {
        const float* part = P.part + ((size_t)row * P.H + h) * kSlices * kPart;
        float dq = 0.0f, dk = 0.0f, da = 0.0f, db = 0.0f;
#pragma unroll
        for (int s = 0; s < kSlices; ++s) {
            dq += part[s * kPart + c];
            dk += part[s * kPart + kDim + c];
            da += part[s * kPart + 2 * kDim + c];
            db += part[s * kPart + 3 * kDim];
        }
        float x;
        const float a = decay(P, row, h, c, eA, &x);
        const float s = sigm(x);
        const float dx = da * a * P.lower_bound * s * (1.0f - s);
        const size_t rk = ((size_t)row * P.H + h) * kDim + c;
        P.dq[rk] = dq;
        P.dk[rk] = dk;
        P.dg[rk] = dx * eA;
        sdg += dx * eA;
        sdA = fmaf(dx, x, sdA);
        if (c == 0) {
            const float sb = sigm(bf(P.beta, (size_t)row * P.H + h));
            P.dbeta[(size_t)row * P.H + h] = db * sb * (1.0f - sb);
        }
    }
    // block sums: dt_bias per key, A_log over the keys (fixed order)
    P.blk[(blk * P.H + h) * (kDim + 1) + c] = sdg;
    for (int o = 16; o > 0; o >>= 1) sdA += __shfl_xor_sync(0xffffffffu, sdA, o);
    if ((c & 31) == 0) red[c >> 5] = sdA;
    __syncthreads();
    if (c == 0) P.blk[(blk * P.H + h) * (kDim + 1) + kDim] = red[0] + red[1] + red[2] + red[3];
}

// dt_bias and A_log gradients: the row blocks summed in order.  One CTA per head.
__global__ void __launch_bounds__(kDim) bwd_reduce_kernel(BwdProblem P, long long nblk,
                                                          const int* valid) {
    if (valid && !*valid) return;
    const int c = threadIdx.x, h = blockIdx.x;
    float s = 0.0f, sA = 0.0f;
    for (long long b = 0; b < nblk; ++b) {
        s += P.blk[(b * P.H + h) * (kDim + 1) + c];
        if (c == 0) sA += P.blk[(b * P.H + h) * (kDim + 1) + kDim];
    }
    P.ddt_bias[(size_t)h * kDim + c] = s;
    if (c == 0) P.dA_log[h] = sA;
}

std::atomic<bool> g_bwd_attr[64];

}  // namespace

size_t bwd_scratch_floats(int N, long long rows, int H, size_t* ck, size_t* fw, size_t* part,
                          size_t* blk) {
    const long long slots = N + rows / kBC + 1;
    *ck = (size_t)slots * H * kSlices * kCkFloats;
    *fw = (size_t)rows * H * kSlices * 2 * kSliceV;
    *part = (size_t)rows * H * kSlices * kPart;
    *blk = (size_t)((rows + kRowBlock - 1) / kRowBlock) * H * (kDim + 1);
    return *ck + *fw + *part + *blk;
}

cudaError_t launch_bwd_main(const BwdProblem& P, const int* valid, cudaStream_t s) {
    const int smem = (int)sizeof(BwdSmem);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !g_bwd_attr[dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) g_bwd_attr[dev].store(true, std::memory_order_release);
    }
    const long long ctas = (long long)P.N * P.H * kSlices;
    if (ctas > 0) bwd_kernel<<<(unsigned)ctas, kBwdThreads, smem, s>>>(P, valid);
    return cudaGetLastError();
}

cudaError_t launch_bwd_finish(const BwdProblem& P, long long rows, const int* valid,
                              cudaStream_t s) {
    const long long nblk = (rows + kRowBlock - 1) / kRowBlock;
    if (nblk > 0) bwd_finish_kernel<<<(unsigned)(nblk * P.H), kDim, 0, s>>>(P, rows, valid);
    return cudaGetLastError();
}

cudaError_t launch_bwd_reduce(const BwdProblem& P, long long rows, const int* valid,
                              cudaStream_t s) {
    const long long nblk = (rows + kRowBlock - 1) / kRowBlock;
    bwd_reduce_kernel<<<(unsigned)P.H, kDim, 0, s>>>(P, nblk, valid);
    return cudaGetLastError();
}

}  // namespace kda
