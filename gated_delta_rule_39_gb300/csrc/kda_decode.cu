// One decode step of KDA: a single new token per (sequence, head) applied to a
// state held in HBM, the step that follows a prefill when the final state is
// used "for efficient incremental decoding" ("FlashKDA", productcool.com,
// "Main Features").  Per (n, h), with the same gate as the prefill:
//
//   gl[c]  = lower_bound * sigmoid(exp(A_log[h]) * (g[c] + dt_bias[h, c]))
//   S'     = Diag(exp(gl)) S                      (row c of S scaled)
//   r      = S'^T k,  delta = b (v - r),  b = sigmoid(beta)
//   S_new  = S' + k delta^T                       (= (I - b k k^T) S' + b k v^T)
//   o      = scale * S_new^T q
//
// The work is the state's 64 KB (fp32) in and out per (n, h): one CTA of eight
// warps per (n, h), warp w owning state rows 16 w .. 16 w + 15 and lane l columns
// 4 l .. 4 l + 3, so that every state access is a 16-byte load or store and a
// warp moves whole 512-byte rows.  Each thread keeps its 64 state values in
// registers from the read to the write, which also makes an in-place update safe.
#include <atomic>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kDecThreads = 256;   // 8 warps x 16 rows
constexpr int kRows = kDim / 8;    // rows per warp

struct DecSmem {
    float alpha[kDim];        // exp(gl) per key channel (row)
    float kq[2][kDim];        // k, q as fp32
    float part[8][kDim];      // per-warp partial sums over its rows (r, then o)
};

__device__ __forceinline__ float4 load_state4(const void* base, int dtype, size_t idx) {
    if (dtype == KDA_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + idx);
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store_state4(void* base, int dtype, size_t idx, float4 x) {
    if (dtype == KDA_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + idx) = x;
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y);
        const __nv_bfloat162 b = __floats2bfloat162_rn(x.z, x.w);
        uint2 raw;
        raw.x = *reinterpret_cast<const uint32_t*>(&a);
        raw.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + idx) = raw;
    }
}

// P.N sequences of one token each; P.init_state / P.final_state are the state in / out
__global__ void __launch_bounds__(kDecThreads) decode_kernel(Problem P) {
    __shared__ DecSmem S;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % P.H;
    const size_t unit = blockIdx.x;                       // n * H + h
    const size_t row_off = unit * kDim;                   // q, k, g, v, out of this (n, h)
    const size_t sbase = unit * kDim * kDim;              // state [n][h][128][128]
    const int c0 = 4 * lane;

    // state rows of this warp (issued first: they are the traffic)
    float4 s[kRows];
    if (P.init_state) {
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            s[i] = load_state4(P.init_state, P.init_dtype, sbase + (size_t)(kRows * w + i) * kDim + c0);
    } else {
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    // gate, k and q of the token
    if (tid < kDim) {
        const float expA = expf(P.A_log[h]);
        const float x = -expA * kLog2e * (__bfloat162float(P.g[row_off + tid]) + P.dt_bias[(size_t)h * kDim + tid]);
        const float sg = rcp_approx(1.0f + ex2_approx(x));           // sigmoid, base 2
        S.alpha[tid] = ex2_approx(P.lower_bound * kLog2e * sg);       // exp(gl)
        S.kq[0][tid] = __bfloat162float(P.k[row_off + tid]);
    } else {
        S.kq[1][tid - kDim] = __bfloat162float(P.q[row_off + tid - kDim]);
    }
    const float b = sigmoid_fast(__bfloat162float(P.beta[unit]));
    const uint2 vraw = *reinterpret_cast<const uint2*>(P.v + row_off + c0);
    const float4 vv = make_float4(__uint_as_float(vraw.x << 16), __uint_as_float(vraw.x & 0xFFFF0000u),
                                  __uint_as_float(vraw.y << 16), __uint_as_float(vraw.y & 0xFFFF0000u));
    __syncthreads();

    // S' = Diag(alpha) S and this warp's part of r = S'^T k
    float4 r = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        const int row = kRows * w + i;
        const float a = S.alpha[row], kr = S.kq[0][row];
        s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
        r.x = fmaf(kr, s[i].x, r.x); r.y = fmaf(kr, s[i].y, r.y);
        r.z = fmaf(kr, s[i].z, r.z); r.w = fmaf(kr, s[i].w, r.w);
    }
    *reinterpret_cast<float4*>(&S.part[w][c0]) = r;
    __syncthreads();
    // r summed over the eight warps in a fixed order; delta = b (v - r)
    float4 rt = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 p = *reinterpret_cast<const float4*>(&S.part[j][c0]);
        rt.x += p.x; rt.y += p.y; rt.z += p.z; rt.w += p.w;
    }
    const float4 dl = make_float4(b * (vv.x - rt.x), b * (vv.y - rt.y), b * (vv.z - rt.z), b * (vv.w - rt.w));
    __syncthreads();   // every warp has read the r partials before they are overwritten

    // S_new = S' + k delta^T, written out; this warp's part of o = S_new^T q
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        const int row = kRows * w + i;
        const float kr = S.kq[0][row], qr = S.kq[1][row];
        s[i].x = fmaf(kr, dl.x, s[i].x); s[i].y = fmaf(kr, dl.y, s[i].y);
        s[i].z = fmaf(kr, dl.z, s[i].z); s[i].w = fmaf(kr, dl.w, s[i].w);
        o.x = fmaf(qr, s[i].x, o.x); o.y = fmaf(qr, s[i].y, o.y);
        o.z = fmaf(qr, s[i].z, o.z); o.w = fmaf(qr, s[i].w, o.w);
        if (P.final_state)
            store_state4(P.final_state, P.final_dtype, sbase + (size_t)row * kDim + c0, s[i]);
    }
    *reinterpret_cast<float4*>(&S.part[w][c0]) = o;
    __syncthreads();
    if (w == 0) {
        float4 ot = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 p = *reinterpret_cast<const float4*>(&S.part[j][c0]);
            ot.x += p.x; ot.y += p.y; ot.z += p.z; ot.w += p.w;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(P.scale * ot.x, P.scale * ot.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(P.scale * ot.z, P.scale * ot.w);
        uint2 raw;
        raw.x = *reinterpret_cast<const uint32_t*>(&lo);
        raw.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(P.out + row_off + c0) = raw;
    }
}

}  // namespace

cudaError_t launch_decode(const Problem& P, cudaStream_t s) {
    const long long ctas = (long long)P.N * P.H;
    if (ctas == 0) return cudaSuccess;
    decode_kernel<<<(unsigned)ctas, kDecThreads, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace kda
