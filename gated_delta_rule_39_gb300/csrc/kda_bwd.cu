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
// each: thread (column j, key block b) holds S[8 b .. 8 b + 7][16 s + j], so a warp
// holds all 128 keys of two columns and the sums over keys (r = S'^T k, dd = dS^T k)
// are four shuffles.  Each block of 8 token rows is staged in shared memory at once.
// Phase 1 runs the slice forward, storing its state every 8 tokens and each token's
// d and v - r; phase 2 walks the blocks backwards, rebuilds the block's states from the
// checkpoint (element-wise, with the stored d) into shared memory, and runs the
// reverse steps.  dq, dk, da and db sum over value columns: within a warp by a
// shuffle, over the 8 warps in shared memory every 2 tokens, and over the 8 slices by
// a second kernel (all in a fixed order), which also applies the activations.
// This is a token-by-token pass on CUDA cores; a chunked pass on tensor cores, as the
// forward is, would be much faster.
#include <atomic>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kSlices = 8;          // value slices per (sequence, head)
constexpr int kSliceV = kDim / kSlices;   // 16 value columns
constexpr int kBwdThreads = 256;    // 128 keys x 2 halves of 8 columns
constexpr int kPart = 388;          // partial sums per (row, head, slice): dq, dk, da [128], db
constexpr int kGroup = 2;           // tokens whose per-warp partial sums wait in shared memory
constexpr int kBC = 8;              // tokens per checkpoint (and per staged block of rows):
                                    // small enough for two CTAs per SM

struct BwdSmem {
    float4 st[kBC][2][kBwdThreads];     // S_{t-1} of each token of the block: a thread's 8
                                        // values as two float4 planes (no bank conflicts)
    float a[kBC][kDim];                  // the block's decays
    float kk[kBC][kDim];                 // keys
    float qq[kBC][kDim];                 // queries (reverse phase)
    float vv[kBC][kSliceV];             // the slice's values (forward) or dL/d(out) (reverse)
    float fw[kBC][2 * kSliceV];         // d and v - r of the slice (reverse)
    float b[kBC];                       // sigmoid(beta)
    // reverse: per-warp sums over the warp's two columns of dq, dk, da (128 keys each)
    // and db, for a group of 4 tokens; summed over the 8 warps once per group
    float grp[kGroup][8][3 * kDim + 4];
};

__device__ __forceinline__ float bf(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }

// the decay of key channel c at token row t, and x (the sigmoid's argument)
__device__ __forceinline__ float decay(const BwdProblem& P, size_t row, int h, int c, float eA,
                                      float* xo = nullptr) {
    const float x = eA * (bf(P.g, (row * P.H + h) * kDim + c) + P.dt_bias[(size_t)h * kDim + c]);
    if (xo) *xo = x;
    return expf(P.lower_bound * sigm(x));
}

// Checkpoint slot of block c (of 8 tokens) of sequence n (first token bos): distinct for
// every (n, c) of a call, below N + rows / 8 + 1.
__device__ __forceinline__ long long ck_slot(int n, long long bos, int c) {
    return (long long)n + c + bos / kBC;
}

// Position of key channel c in the staged rows and in the per-warp column sums: the 8
// keys of key block kb = c / 8 sit in two planes, keys 0-3 at 4 kb and keys 4-7 at
// 64 + 4 kb, so that the 16 key blocks of a warp read or write 16 consecutive float4 per
// plane (no bank conflicts).  kkey is the inverse.
__device__ __forceinline__ int kpos(int c) { return ((c & 4) << 4) + ((c >> 3) << 2) + (c & 3); }
__device__ __forceinline__ int kkey(int p) { return ((p & 63) >> 2) * 8 + ((p >> 6) << 2) + (p & 3); }

// A block's raw token rows, loaded into registers one block ahead of their use, so that
// their memory latency overlaps the block before: keys, gate inputs (and queries on the
// way back) as thread (row, 4 channels); in x, the slice's 16 values or dL/d(out)
// (threads 0-15, 8 columns each), the beta logit (threads 16-23) or the stored d and
// v - r on the way back (threads 128-191, 4 floats each).  Rows past the sequence's end
// are not read.
struct Rows {
    uint2 k, g, q;
    uint4 x;
};

__device__ __forceinline__ void fetch(const BwdProblem& P, Rows& R, long long row0, int len,
                                      int h, int col0, bool reverse, const float* fw0,
                                      size_t fw_step) {
    const int tid = threadIdx.x;
    const int i = tid >> 5, c4 = 4 * (tid & 31);
    if (i < len) {
        const size_t rk = ((size_t)(row0 + i) * P.H + h) * kDim + c4;
        R.k = *reinterpret_cast<const uint2*>(P.k + rk);
        R.g = *reinterpret_cast<const uint2*>(P.g + rk);
        if (reverse) R.q = *reinterpret_cast<const uint2*>(P.q + rk);
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
    } else if (reverse && tid >= 128 && tid < 128 + 8 * kBC) {
        const int r = (tid - 128) >> 3, f4 = 4 * ((tid - 128) & 7);
        if (r < len) R.x = *reinterpret_cast<const uint4*>(fw0 + (size_t)r * fw_step + f4);
    }
}

__device__ __forceinline__ void unpack4(uint2 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xFFFF0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xFFFF0000u);
}

// The fetched rows into shared memory (decays and b formed on the way), then a barrier.
// dtb: dt_bias of the thread's 4 channels.
__device__ __forceinline__ void commit(BwdSmem& S, const Rows& R, int len, float eA,
                                       float lower_bound, const float (&dtb)[4], bool reverse) {
    const int tid = threadIdx.x;
    const int i = tid >> 5, p = kpos(4 * (tid & 31));
    if (i < len) {
        float kx[4], gx[4], a[4];
        unpack4(R.k, kx);
        unpack4(R.g, gx);
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = expf(lower_bound * sigm(eA * (gx[e] + dtb[e])));
        *reinterpret_cast<float4*>(&S.a[i][p]) = make_float4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<float4*>(&S.kk[i][p]) = make_float4(kx[0], kx[1], kx[2], kx[3]);
        if (reverse) {
            float qx[4];
            unpack4(R.q, qx);
            *reinterpret_cast<float4*>(&S.qq[i][p]) = make_float4(qx[0], qx[1], qx[2], qx[3]);
        }
    }
    if (tid < 2 * kBC) {
        const int r = tid >> 1, hv = tid & 1;
        if (r < len) {
            float lo[4], hi[4];
            unpack4(make_uint2(R.x.x, R.x.y), lo);
            unpack4(make_uint2(R.x.z, R.x.w), hi);
            *reinterpret_cast<float4*>(&S.vv[r][8 * hv]) = make_float4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<float4*>(&S.vv[r][8 * hv + 4]) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        }
    } else if (tid < 3 * kBC) {
        const int r = tid - 2 * kBC;
        if (r < len) S.b[r] = sigm(__uint_as_float(R.x.x));
    } else if (reverse && tid >= 128 && tid < 128 + 8 * kBC) {
        const int r = (tid - 128) >> 3, f4 = 4 * ((tid - 128) & 7);
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
__device__ __forceinline__ float2 shfl16(float2 a) {
    return make_float2(__shfl_xor_sync(0xffffffffu, a.x, 16), __shfl_xor_sync(0xffffffffu, a.y, 16));
}

// A thread's 8 keys of a staged row (or of a column-sum row) as 4 pairs: keys 8 kb + 0-3
// from the first plane, 4-7 from the second.
__device__ __forceinline__ void ld_planes(const float* row, int pk, float2 (&x)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(row + pk);
    const float4 w = *reinterpret_cast<const float4*>(row + 64 + pk);
    x[0] = make_float2(u.x, u.y); x[1] = make_float2(u.z, u.w);
    x[2] = make_float2(w.x, w.y); x[3] = make_float2(w.z, w.w);
}

__device__ __forceinline__ void st_planes(float* row, int pk, const float2 (&x)[4]) {
    *reinterpret_cast<float4*>(row + pk) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
    *reinterpret_cast<float4*>(row + 64 + pk) = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
}

__global__ void __launch_bounds__(kBwdThreads, 2) bwd_kernel(BwdProblem P, const int* valid) {
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
    const float eA = expf(P.A_log[h]);
    const size_t fw_step = (size_t)P.H * kSlices * (2 * kSliceV);           // between rows
    const auto fw_at = [&](size_t row) {   // d (16) and v - r (16) of this slice at a row
        return P.fw + ((row * P.H + h) * kSlices + slice) * (2 * kSliceV);
    };
    const auto ck_at = [&](int c) {        // checkpoint of block c: [key][16 columns]
        return P.ck + ((ck_slot(n, bos, c) * P.H + h) * kSlices + slice) * (kDim * kSliceV);
    };
    float dtb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) dtb[e] = P.dt_bias[(size_t)h * kDim + 4 * (tid & 31) + e];
    // Thread (column jv = tid / 16, key block kb = tid % 16) holds S[8 kb .. + 7][jv] in
    // both phases: a warp holds all 128 keys of two columns, so r = S'^T k and dd = dS^T k
    // are sums over 16 lanes (four shuffles, no barrier per token).
    const int jv = tid >> 4, kb = tid & 15, k0 = 8 * kb, pk = 4 * kb;
    Rows R{};

    // ---- phase 1: forward over the slice, checkpoints and per-token d, v - r ----------
    {
        float2 st[4];   // keys k0 + 2e, k0 + 2e + 1
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float x = 0.0f;
            if (P.init_state) {
                const size_t si = (((size_t)n * P.H + h) * kDim + k0 + e) * kDim + col0 + jv;
                x = P.init_dtype == KDA_F32 ? static_cast<const float*>(P.init_state)[si]
                                            : __bfloat162float(static_cast<const __nv_bfloat16*>(P.init_state)[si]);
            }
            if (e & 1) st[e >> 1].y = x; else st[e >> 1].x = x;
        }
        if (nch > 0) fetch(P, R, bos, min(kBC, L), h, col0, false, nullptr, 0);
        for (int c = 0; c < nch; ++c) {
            float* ck = ck_at(c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ck[(k0 + 2 * e) * kSliceV + jv] = st[e].x;
                ck[(k0 + 2 * e + 1) * kSliceV + jv] = st[e].y;
            }
            const int len = min(kBC, L - c * kBC);
            const long long row0 = bos + (long long)c * kBC;
            commit(S, R, len, eA, P.lower_bound, dtb, false);
            if (c + 1 < nch)
                fetch(P, R, row0 + kBC, min(kBC, L - (c + 1) * kBC), h, col0, false, nullptr, 0);
            for (int i = 0; i < len; ++i) {
                float2 a[4], kk[4], r2 = make_float2(0.0f, 0.0f);
                ld_planes(S.a[i], pk, a);
                ld_planes(S.kk[i], pk, kk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    st[e] = mul2(st[e], a[e]);
                    r2 = fma2(st[e], kk[e], r2);
                }
                float r = r2.x + r2.y;
                r += __shfl_xor_sync(0xffffffffu, r, 1);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                r += __shfl_xor_sync(0xffffffffu, r, 4);
                r += __shfl_xor_sync(0xffffffffu, r, 8);
                const float vr = S.vv[i][jv] - r;
                const float d = S.b[i] * vr;
#pragma unroll
                for (int e = 0; e < 4; ++e) st[e] = fma2(kk[e], dup2(d), st[e]);
                if (kb == 0) {   // lanes 0 and 16: this column's d and v - r
                    float* f = fw_at(row0 + i);
                    f[jv] = d;
                    f[kSliceV + jv] = vr;
                }
            }
            __syncthreads();   // the staged rows are replaced by the next block's
        }
    }
    __syncthreads();   // d and v - r are read by other threads below

    // ---- phase 2: reverse, block by block from the last ---------------------------------
    float2 dS[4];
    float ckn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float x =
            P.dfinal ? P.dfinal[(((size_t)n * P.H + h) * kDim + k0 + e) * kDim + col0 + jv] : 0.0f;
        if (e & 1) dS[e >> 1].y = x; else dS[e >> 1].x = x;
    }
    if (nch > 0) {
        const long long row0 = bos + (long long)(nch - 1) * kBC;
        fetch(P, R, row0, L - (nch - 1) * kBC, h, col0, true, fw_at(row0), fw_step);
        const float* ck = ck_at(nch - 1);
#pragma unroll
        for (int e = 0; e < 8; ++e) ckn[e] = ck[(k0 + e) * kSliceV + jv];   // written by this thread
    }
    for (int c = nch - 1; c >= 0; --c) {
        const int len = min(kBC, L - c * kBC);
        const long long row0 = bos + (long long)c * kBC;
        commit(S, R, len, eA, P.lower_bound, dtb, true);
        float2 sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sv[e] = make_float2(ckn[2 * e], ckn[2 * e + 1]);
        if (c > 0) {   // the block before is whole
            fetch(P, R, row0 - kBC, kBC, h, col0, true, fw_at(row0 - kBC), fw_step);
            const float* ck = ck_at(c - 1);
#pragma unroll
            for (int e = 0; e < 8; ++e) ckn[e] = ck[(k0 + e) * kSliceV + jv];
        }
        // rebuild the block's states S_{t-1} from the checkpoint (element-wise, the same
        // arithmetic as phase 1; each thread reads back only its own states)
        for (int i = 0; i < len; ++i) {
            S.st[i][0][tid] = make_float4(sv[0].x, sv[0].y, sv[1].x, sv[1].y);
            S.st[i][1][tid] = make_float4(sv[2].x, sv[2].y, sv[3].x, sv[3].y);
            const float d = S.fw[i][jv];
            float2 a[4], kk[4];
            ld_planes(S.a[i], pk, a);
            ld_planes(S.kk[i], pk, kk);
#pragma unroll
            for (int e = 0; e < 4; ++e) sv[e] = fma2(kk[e], dup2(d), mul2(sv[e], a[e]));
        }
        for (int i = len - 1; i >= 0; --i) {
            const int gi = (len - 1 - i) % kGroup;   // slot of this token in its group
            float2 a[4], kk[4], qq[4];
            ld_planes(S.a[i], pk, a);
            ld_planes(S.kk[i], pk, kk);
            ld_planes(S.qq[i], pk, qq);
            const float d = S.fw[i][jv], vr = S.fw[i][kSliceV + jv];
            const float dout = S.vv[i][jv], b = S.b[i];
            const float4 p0 = S.st[i][0][tid];
            const float4 p1 = S.st[i][1][tid];
            const float2 sprev[4] = {make_float2(p0.x, p0.y), make_float2(p0.z, p0.w),
                                     make_float2(p1.x, p1.y), make_float2(p1.z, p1.w)};
            float2 sp[4], dq[4], dk[4], da[4], dd2 = make_float2(0.0f, 0.0f);
            const float2 d2 = dup2(d), do2 = dup2(dout), sdo2 = dup2(P.scale * dout);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sp[e] = mul2(sprev[e], a[e]);
                dq[e] = mul2(fma2(kk[e], d2, sp[e]), do2);   // S_t dO (scale applied at the end)
                dS[e] = fma2(qq[e], sdo2, dS[e]);
                dk[e] = mul2(dS[e], d2);
                dd2 = fma2(dS[e], kk[e], dd2);
            }
            float dd = dd2.x + dd2.y;
            dd += __shfl_xor_sync(0xffffffffu, dd, 1);   // dd = dS^T k over the 128 keys
            dd += __shfl_xor_sync(0xffffffffu, dd, 2);
            dd += __shfl_xor_sync(0xffffffffu, dd, 4);
            dd += __shfl_xor_sync(0xffffffffu, dd, 8);
            const float2 dr2 = dup2(-b * dd);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 dsp = fma2(kk[e], dr2, dS[e]);
                dk[e] = fma2(sp[e], dr2, dk[e]);
                da[e] = mul2(dsp, sprev[e]);
                dS[e] = mul2(a[e], dsp);
            }
            float db = dd * vr;
            const size_t row = row0 + i;
            if (kb == 0) P.dv[(row * P.H + h) * kDim + col0 + jv] = b * dd;
            // the warp's two columns (lanes l and l ^ 16) added, then kept for the group
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dq[e] = add2(dq[e], shfl16(dq[e]));
                dk[e] = add2(dk[e], shfl16(dk[e]));
                da[e] = add2(da[e], shfl16(da[e]));
            }
            db += __shfl_xor_sync(0xffffffffu, db, 16);
            if (lane < 16) {
                float* gp = S.grp[gi][warp];
                st_planes(gp, pk, dq);
                st_planes(gp + kDim, pk, dk);
                st_planes(gp + 2 * kDim, pk, da);
                if (lane == 0) gp[3 * kDim] = db;
            }
            if (gi == kGroup - 1 || i == 0) {
                // the group's tokens (rows row .. row + gi): sum the 8 warps in order and
                // write this slice's partial sums in key order
                __syncthreads();
                for (int g = 0; g <= gi; ++g) {
                    const size_t grow = row + gi - g;   // slot g holds the g-th token walked
                    float* out = P.part + ((grow * P.H + h) * kSlices + slice) * kPart;
                    for (int e2 = tid; e2 <= 3 * kDim / 2; e2 += kBwdThreads) {   // pairs
                        const int e = 2 * e2;
                        float2 sum = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int w = 0; w < 8; ++w)
                            sum = add2(sum, *reinterpret_cast<const float2*>(&S.grp[g][w][e]));
                        const int sec = e >> 7;   // dq, dk, da; the last pair holds db
                        if (sec == 3) {
                            out[3 * kDim] = sum.x;
                        } else {   // positions e, e + 1 are keys kkey(e), kkey(e) + 1
                            *reinterpret_cast<float2*>(out + sec * kDim + kkey(e & (kDim - 1))) =
                                sec == 0 ? mul2(sum, dup2(P.scale)) : sum;
                        }
                    }
                }
                __syncthreads();
            }
        }
        __syncthreads();   // the block's staged rows and states are replaced by the next one
    }
    if (P.d_init) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            P.d_init[(((size_t)n * P.H + h) * kDim + k0 + e) * kDim + col0 + jv] =
                (e & 1) ? dS[e >> 1].y : dS[e >> 1].x;
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
    *ck = (size_t)slots * H * kSlices * kDim * kSliceV;
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
