// kda_decode.cu -- the recurrent decode step: a few tokens (typically one) per
// (sequence, head), applied to a resident state with fp32 or bf16 storage.
//
// Per token (the gated delta rule with per-channel decay, cuLA PR #103 "feat(kda/sm90):
// FlashKDA prefill port + intracard-CP prefill", problem statement; the same
// recurrence the prefill computes chunkwise):
//     S' = Diag(exp g) S,   u = S'^T k,   delta = beta (v - u),
//     S  = S' + k delta^T,  o = scale S^T q = scale (S'^T q + (q . k) delta).
// The last form needs one pass over the state for both reductions (u and S'^T q);
// the update is the second pass, over the same registers.
//
// HBM-bound: each (sequence, head) reads its 128 x 128 state once and writes it once
// (64 KiB each way in fp32, 32 KiB in bf16); per token only q, k, v, g, beta and the
// output row move.  One 256-thread CTA per (sequence, head): warp w holds key rows
// 16w .. 16w + 15, lane l value columns 4l .. 4l + 3, so a warp's load of one state row
// is 512 contiguous bytes (fp32) and the state sits in 64 registers per thread.  The
// reductions over key rows finish in shared memory across the 8 warps.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecRows = 16;  // key rows per warp

__device__ __forceinline__ void state_load(const float* p, float (&x)[4]) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void state_load(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
__device__ __forceinline__ void state_store(float* p, const float (&x)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
}
__device__ __forceinline__ void state_store(__nv_bfloat16* p, const float (&x)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&a);
    v.y = *reinterpret_cast<const uint32_t*>(&b);
    __stcs(reinterpret_cast<uint2*>(p), v);
}

template <typename ST>
__global__ void __launch_bounds__(kDecThreads, 2) kda_decode_kernel(const DecodeParams p) {
    __shared__ float s_k[kD], s_q[kD], s_e[kD], s_v[kD], s_d[kD];
    __shared__ __align__(16) float s_red[2][kDecThreads / 32][kD];
    __shared__ float s_qk[kDecThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t nh = blockIdx.x;
    const int64_t n = nh / p.H;
    const int h = (int)(nh % p.H);
    const int r0 = warp * kDecRows, c0 = lane * 4;
    const size_t soff = (size_t)nh * kD * kD + (size_t)r0 * kD + c0;

    float s[kDecRows][4];
    if (p.s0) {
        const ST* src = static_cast<const ST*>(p.s0) + soff;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) state_load(src + (size_t)r * kD, s[r]);
    } else {
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) s[r][0] = s[r][1] = s[r][2] = s[r][3] = 0.f;
    }

    // Row (token t, head h) of sequence n starts at element (n T + t) H + h.  Threads
    // 0..127 stage one channel each of the token's q, k, v and exp(g).
    const size_t row0 = (size_t)n * p.T * p.H + h;
    for (int64_t t = 0; t < p.T; ++t) {
        const size_t row = row0 + (size_t)t * p.H;
        float beta_t = 0.f;
        if (tid < kD) {
            const size_t e = row * kD + tid;
            s_k[tid] = __bfloat162float(p.k[e]);
            s_q[tid] = __bfloat162float(p.q[e]);
            s_v[tid] = __bfloat162float(p.v[e]);
            s_e[tid] = expf(p.g[e]);
            beta_t = __bfloat162float(p.beta[row]);
        }
        __syncthreads();

        // Pass 1: decay the rows, partial u = S'^T k and w = S'^T q over this warp's rows.
        float u[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f}, qk = 0.f;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) {
            const float e = s_e[r0 + r], kr = s_k[r0 + r], qr = s_q[r0 + r];
            qk = fmaf(qr, kr, qk);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                s[r][c] *= e;
                u[c] = fmaf(kr, s[r][c], u[c]);
                w[c] = fmaf(qr, s[r][c], w[c]);
            }
        }
        *reinterpret_cast<float4*>(&s_red[0][warp][c0]) = make_float4(u[0], u[1], u[2], u[3]);
        *reinterpret_cast<float4*>(&s_red[1][warp][c0]) = make_float4(w[0], w[1], w[2], w[3]);
        if (lane == 0) s_qk[warp] = qk;
        __syncthreads();

        // Column j = tid: delta_j and the output o_j.
        if (tid < kD) {
            float uu = 0.f, ww = 0.f, qq = 0.f;
#pragma unroll
            for (int x = 0; x < kDecThreads / 32; ++x) {
                uu += s_red[0][x][tid];
                ww += s_red[1][x][tid];
                qq += s_qk[x];
            }
            const float d = beta_t * (s_v[tid] - uu);
            s_d[tid] = d;
            p.out[row * kD + tid] = __float2bfloat16_rn(p.scale * fmaf(qq, d, ww));
        }
        __syncthreads();

        // Pass 2: S = S' + k delta^T.
        const float4 d4 = *reinterpret_cast<const float4*>(&s_d[c0]);
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) {
            const float kr = s_k[r0 + r];
            s[r][0] = fmaf(kr, d4.x, s[r][0]);
            s[r][1] = fmaf(kr, d4.y, s[r][1]);
            s[r][2] = fmaf(kr, d4.z, s[r][2]);
            s[r][3] = fmaf(kr, d4.w, s[r][3]);
        }
        // The next token overwrites s_k / s_d only after every warp has passed here.
        if (t + 1 < p.T) __syncthreads();
    }

    if (p.sfin) {
        ST* dst = static_cast<ST*>(p.sfin) + soff;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) state_store(dst + (size_t)r * kD, s[r]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.N * p.H;
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)rows), block(kDecThreads);
    if (p.state_bf16)
        kda_decode_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(p);
    else
        kda_decode_kernel<float><<<grid, block, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
