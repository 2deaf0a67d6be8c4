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
// each: thread (key c, half h) holds S[c][16 s + 8 h .. + 7].  Phase 1 runs the slice
// forward, storing its state every 16 tokens and each token's d and v - r; phase 2
// walks the chunks backwards, rebuilds the chunk's states from the checkpoint
// (element-wise, with the stored d) into shared memory, and runs the reverse steps.
// dq, dk, da and db sum over value columns: each slice writes its partial sums, and a
// second kernel adds the 8 slices in a fixed order and applies the activations.
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

struct BwdSmem {
    float st[kChunk][kBwdThreads][8];   // S_{t-1} of each token of the chunk, per thread
    float red[2][8][kSliceV];           // warp partials of the key reductions (two buffers)
};

__device__ __forceinline__ float bf(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }

// x[e] summed over the 128 keys (threads of the same half), for this thread's 8 columns
__device__ __forceinline__ void key_sum(float (&x)[8], BwdSmem& S, int buf, int warp, int lane) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float y = x[e];
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        y += __shfl_xor_sync(0xffffffffu, y, 4);
        y += __shfl_xor_sync(0xffffffffu, y, 8);
        y += __shfl_xor_sync(0xffffffffu, y, 16);
        x[e] = y;
    }
    if (lane < 2) {
        float* r = &S.red[buf][warp][8 * lane];
        *reinterpret_cast<float4*>(r) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(r + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    const int hv = lane & 1;
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const float4 p = *reinterpret_cast<const float4*>(&S.red[buf][w][8 * hv]);
        const float4 q = *reinterpret_cast<const float4*>(&S.red[buf][w][8 * hv + 4]);
        x[0] += p.x; x[1] += p.y; x[2] += p.z; x[3] += p.w;
        x[4] += q.x; x[5] += q.y; x[6] += q.z; x[7] += q.w;
    }
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }

// the decay of key channel c at token row t, and x (the sigmoid's argument)
__device__ __forceinline__ float decay(const BwdProblem& P, size_t row, int h, int c, float eA,
                                      float* xo = nullptr) {
    const float x = eA * (bf(P.g, (row * P.H + h) * kDim + c) + P.dt_bias[(size_t)h * kDim + c]);
    if (xo) *xo = x;
    return expf(P.lower_bound * sigm(x));
}

// Checkpoint slot of chunk c of sequence n (first token bos): distinct for every
// (n, c) of a call, below N + rows / 16 + 1.
__device__ __forceinline__ long long ck_slot(int n, long long bos, int c) {
    return (long long)n + c + bos / kChunk;
}

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(BwdProblem P, const int* valid) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem& S = *reinterpret_cast<BwdSmem*>(smem_raw);
    if (valid && !*valid) return;   // malformed cu_seqlens: the sequence map says so
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int key = tid >> 1, hv = tid & 1;
    const int slice = blockIdx.x % kSlices;
    const int h = (blockIdx.x / kSlices) % P.H;
    const int n = blockIdx.x / (kSlices * P.H);
    const long long bos = P.cu_seqlens ? P.cu_seqlens[n] : (long long)n * P.T;
    const int L = P.cu_seqlens ? P.cu_seqlens[n + 1] - P.cu_seqlens[n] : P.T;
    const int nch = (L + kChunk - 1) / kChunk;
    const int col = kSliceV * slice + 8 * hv;                  // first of this thread's columns
    const float eA = expf(P.A_log[h]);
    const size_t sidx = (((size_t)n * P.H + h) * kDim + key) * kDim + col;   // state element
    const auto fw_at = [&](size_t row) {   // d (16) and v - r (16) of this slice at a row
        return P.fw + ((row * P.H + h) * kSlices + slice) * (2 * kSliceV);
    };
    const auto ck_at = [&](int c) {
        return P.ck + ((ck_slot(n, bos, c) * P.H + h) * kSlices + slice) * (kDim * kSliceV) +
               key * kSliceV + 8 * hv;
    };

    // ---- phase 1: forward over the slice, checkpoints and per-token d, v - r ----------
    float st[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float x = 0.0f;
        if (P.init_state)
            x = P.init_dtype == KDA_F32 ? static_cast<const float*>(P.init_state)[sidx + e]
                                        : __bfloat162float(static_cast<const __nv_bfloat16*>(P.init_state)[sidx + e]);
        st[e] = x;
    }
    int buf = 0;
    for (int c = 0; c < nch; ++c) {
        float* ck = ck_at(c);
        *reinterpret_cast<float4*>(ck) = make_float4(st[0], st[1], st[2], st[3]);
        *reinterpret_cast<float4*>(ck + 4) = make_float4(st[4], st[5], st[6], st[7]);
        const int len = min(kChunk, L - c * kChunk);
        for (int i = 0; i < len; ++i) {
            const size_t row = bos + (size_t)c * kChunk + i;
            const float a = decay(P, row, h, key, eA);
            const float kk = bf(P.k, (row * P.H + h) * kDim + key);
            const float b = sigm(bf(P.beta, row * P.H + h));
            float vv[8], r[8];
            load8_bf16(P.v + (row * P.H + h) * kDim + col, vv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                st[e] *= a;
                r[e] = st[e] * kk;
            }
            key_sum(r, S, buf, warp, lane);
            buf ^= 1;
            float d[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                d[e] = b * (vv[e] - r[e]);
                st[e] = fmaf(kk, d[e], st[e]);
            }
            if (key == 0) {   // threads 0 and 1: the 16 columns of the slice
                float* f = fw_at(row) + 8 * hv;
                *reinterpret_cast<float4*>(f) = make_float4(d[0], d[1], d[2], d[3]);
                *reinterpret_cast<float4*>(f + 4) = make_float4(d[4], d[5], d[6], d[7]);
                float* g = fw_at(row) + kSliceV + 8 * hv;
                *reinterpret_cast<float4*>(g) = make_float4(vv[0] - r[0], vv[1] - r[1], vv[2] - r[2], vv[3] - r[3]);
                *reinterpret_cast<float4*>(g + 4) = make_float4(vv[4] - r[4], vv[5] - r[5], vv[6] - r[6], vv[7] - r[7]);
            }
        }
    }
    __syncthreads();   // the per-token d and v - r are read by other threads below

    // ---- phase 2: reverse ------------------------------------------------------------
    float dS[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) dS[e] = P.dfinal ? P.dfinal[sidx + e] : 0.0f;
    for (int c = nch - 1; c >= 0; --c) {
        const int len = min(kChunk, L - c * kChunk);
        {   // rebuild the chunk's states S_{t-1} from the checkpoint (element-wise)
            const float* ck = ck_at(c);
            const float4 c0 = *reinterpret_cast<const float4*>(ck);
            const float4 c1 = *reinterpret_cast<const float4*>(ck + 4);
            float s[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            for (int i = 0; i < len; ++i) {
                const size_t row = bos + (size_t)c * kChunk + i;
                *reinterpret_cast<float4*>(&S.st[i][tid][0]) = make_float4(s[0], s[1], s[2], s[3]);
                *reinterpret_cast<float4*>(&S.st[i][tid][4]) = make_float4(s[4], s[5], s[6], s[7]);
                const float a = decay(P, row, h, key, eA);
                const float kk = bf(P.k, (row * P.H + h) * kDim + key);
                const float* f = fw_at(row) + 8 * hv;
                const float4 d0 = *reinterpret_cast<const float4*>(f);
                const float4 d1 = *reinterpret_cast<const float4*>(f + 4);
                const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = fmaf(kk, d[e], a * s[e]);
            }
        }
        // (each thread reads only its own rebuilt states and its own key's decay)
        for (int i = len - 1; i >= 0; --i) {
            const size_t row = bos + (size_t)c * kChunk + i;
            const size_t rk = (row * P.H + h) * kDim;
            const float a = decay(P, row, h, key, eA);
            const float kk = bf(P.k, rk + key), qq = bf(P.q, rk + key);
            const float b = sigm(bf(P.beta, row * P.H + h));
            float dout[8];
            load8_bf16(P.dout + rk + col, dout);
            const float* f = fw_at(row) + 8 * hv;
            const float4 d0 = *reinterpret_cast<const float4*>(f);
            const float4 d1 = *reinterpret_cast<const float4*>(f + 4);
            const float4 w0 = *reinterpret_cast<const float4*>(f + kSliceV);
            const float4 w1 = *reinterpret_cast<const float4*>(f + kSliceV + 4);
            const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            const float vr[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float sp[8], sprev[8];
            {
                const float4 p0 = *reinterpret_cast<const float4*>(&S.st[i][tid][0]);
                const float4 p1 = *reinterpret_cast<const float4*>(&S.st[i][tid][4]);
                sprev[0] = p0.x; sprev[1] = p0.y; sprev[2] = p0.z; sprev[3] = p0.w;
                sprev[4] = p1.x; sprev[5] = p1.y; sprev[6] = p1.z; sprev[7] = p1.w;
            }
            float dq = 0.0f, dk = 0.0f, da = 0.0f;
            float dd[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                sp[e] = a * sprev[e];
                const float snow = fmaf(kk, d[e], sp[e]);
                dS[e] = fmaf(P.scale * qq, dout[e], dS[e]);
                dq = fmaf(snow, dout[e], dq);
                dk = fmaf(dS[e], d[e], dk);
                dd[e] = dS[e] * kk;
            }
            key_sum(dd, S, buf, warp, lane);
            buf ^= 1;
            float db = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                db = fmaf(dd[e], vr[e], db);
                const float dr = -b * dd[e];
                const float dsp = fmaf(kk, dr, dS[e]);
                dk = fmaf(sp[e], dr, dk);
                da = fmaf(dsp, sprev[e], da);
                dS[e] = a * dsp;
            }
            if (key == 0) {   // dv of the slice's 16 columns
                float* o = P.dv + rk + col;
                *reinterpret_cast<float4*>(o) = make_float4(b * dd[0], b * dd[1], b * dd[2], b * dd[3]);
                *reinterpret_cast<float4*>(o + 4) = make_float4(b * dd[4], b * dd[5], b * dd[6], b * dd[7]);
            }
            // the two halves of a key: add their partial sums
            dq += __shfl_xor_sync(0xffffffffu, dq, 1);
            dk += __shfl_xor_sync(0xffffffffu, dk, 1);
            da += __shfl_xor_sync(0xffffffffu, da, 1);
            db += __shfl_xor_sync(0xffffffffu, db, 1);
            float* part = P.part + ((row * P.H + h) * kSlices + slice) * kPart;
            if (hv == 0) {
                part[key] = P.scale * dq;
                part[kDim + key] = dk;
                part[2 * kDim + key] = da;
            }
            if (tid == 0) part[3 * kDim] = db;
        }
        __syncthreads();   // the chunk's rebuilt states are overwritten by the next one
    }
    if (P.d_init) {
        float* o = P.d_init + sidx;
        *reinterpret_cast<float4*>(o) = make_float4(dS[0], dS[1], dS[2], dS[3]);
        *reinterpret_cast<float4*>(o + 4) = make_float4(dS[4], dS[5], dS[6], dS[7]);
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
    const long long slots = N + rows / kChunk + 1;
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
