// kda_decode.cu -- the recurrent decode step: a few tokens (typically one) per
// (sequence, head), applied to a resident state with fp32 or bf16 storage.
//
// Per token (Kimi Delta Attention: the gated delta rule with a per-channel decay, the
// method cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP prefill"
// computes chunkwise; the same recurrence the prefill computes):
//     S' = Diag(exp g) S,   u = S'^T k,   delta = beta (v - u),
//     S  = S' + k delta^T,  o = scale S^T q = scale (S'^T q + (q . k) delta).
// The last form needs one pass over the state for both reductions (u and S'^T q);
// the update is the second pass, over the same registers.
//
// HBM-bound: each (sequence, head) reads its 128 x 128 state once and writes it once
// (64 KiB each way in fp32, 32 KiB in bf16); per token only q, k, v, g, beta and the
// output row move.  fp32 state: one 256-thread CTA per (sequence, head); warp w holds
// key rows 16w .. 16w + 15, lane l value columns 4l .. 4l + 3, so a warp's load of one
// state row is 512 contiguous bytes and the state sits in 64 registers per thread; two
// CTAs per SM keep 128 KiB of loads in flight.  The reductions over key rows finish in
// shared memory across the warps.  bf16 state: its own kernel below.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecRows = 16;  // key rows per warp

__device__ __forceinline__ void state_load(const float* p, float (&x)[4]) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void state_store(float* p, const float (&x)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
}
// kGrouped: unequal head counts (HeadMap); the equal-count instance keeps plain head
// indexing (the map's arithmetic costs the bf16 kernel spills at its register cap).
template <bool kGrouped>
__global__ void __launch_bounds__(kDecThreads, 2) kda_decode_kernel(const DecodeParams p) {
    __shared__ float s_k[kD], s_q[kD], s_e[kD], s_v[kD], s_d[kD];
    __shared__ __align__(16) float s_red[2][kDecThreads / 32][kD];
    __shared__ float s_qk[kDecThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hq = kGrouped ? p.Hq : p.H;
    const int Ho = Hq > p.H ? Hq : p.H, Hk = Hq > p.H ? p.H : Hq;
    const int64_t n = (int64_t)blockIdx.x / Ho;
    const int ho = (int)(blockIdx.x % Ho);
    const HeadMap hm = kGrouped ? head_map(ho, p.H, Hq) : HeadMap{ho, ho, ho, true};
    const int r0 = warp * kDecRows, c0 = lane * 4;
    const size_t soff = ((size_t)n * p.H + hm.hs) * kD * kD + (size_t)r0 * kD + c0;

    float s[kDecRows][4];
    if (p.s0) {
        const float* src = static_cast<const float*>(p.s0) + soff;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) state_load(src + (size_t)r * kD, s[r]);
    } else {
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) s[r][0] = s[r][1] = s[r][2] = s[r][3] = 0.f;
    }

    // Token t of sequence n is token n T + t; a tensor with X heads holds head x of it at
    // row (n T + t) X + x.  Threads 0..127 stage one channel each of q, k, v and exp(g).
    for (int64_t t = 0; t < p.T; ++t) {
        const size_t tok = (size_t)n * p.T + t;
        const size_t row = tok * p.H + hm.hs;
        float beta_t = 0.f;
        if (tid < kD) {
            s_k[tid] = __bfloat162float(p.k[(tok * Hk + hm.hk) * kD + tid]);
            s_q[tid] = __bfloat162float(p.q[(tok * Hq + hm.hq) * kD + tid]);
            s_v[tid] = __bfloat162float(p.v[row * kD + tid]);
            s_e[tid] = expf(p.g[row * kD + tid]);
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
            p.out[(tok * Ho + ho) * kD + tid] = __float2bfloat16_rn(p.scale * fmaf(qq, d, ww));
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

    if (p.sfin && hm.state_owner) {
        float* dst = static_cast<float*>(p.sfin) + soff;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) state_store(dst + (size_t)r * kD, s[r]);
    }
}

// bf16 state storage.  The state stays packed (two bf16 per register), so one thread
// holds 128 elements and a 128-thread CTA covers a head: warp w owns key rows
// 32w .. 32w + 31, half-warp hw = lane / 16 the rows of parity hw among them, lane
// l % 16 value columns 8(l % 16) .. +7.  A warp's 16-byte loads cover two whole rows
// (512 contiguous bytes).  Three CTAs per SM (168 registers a thread) keep 96 KiB of
// state loads in flight per SM, which the bf16 step needs to reach the HBM copy rate
// (two CTAs reach 0.87 of it; four force heavy spills).  Arithmetic is fp32; the state
// is rounded to bf16 after every token, so a T-token call equals T one-token calls bit
// for bit.
constexpr int kDecB16Threads = 128;
constexpr int kDecB16Rows = 16;  // rows per thread

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool kGrouped>
__global__ void __launch_bounds__(kDecB16Threads, 3) kda_decode_bf16_kernel(const DecodeParams p) {
    __shared__ float s_k[kD], s_q[kD], s_e[kD], s_v[kD];
    __shared__ __align__(16) float s_d[kD];
    __shared__ __align__(16) float s_red[2][kDecB16Threads / 32][kD];
    __shared__ float s_qk[kDecB16Threads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hw = lane >> 4, c0 = (lane & 15) * 8;
    const int Hq = kGrouped ? p.Hq : p.H;
    const int Ho = Hq > p.H ? Hq : p.H, Hk = Hq > p.H ? p.H : Hq;
    const int64_t n = (int64_t)blockIdx.x / Ho;
    const int ho = (int)(blockIdx.x % Ho);
    const HeadMap hm = kGrouped ? head_map(ho, p.H, Hq) : HeadMap{ho, ho, ho, true};
    const int rbase = warp * 32 + hw;  // this thread's rows: rbase + 2 i
    const size_t soff = ((size_t)n * p.H + hm.hs) * kD * kD + (size_t)rbase * kD + c0;

    uint4 s[kDecB16Rows];
    if (p.s0) {
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.s0) + soff;
#pragma unroll
        for (int i = 0; i < kDecB16Rows; ++i)
            s[i] = __ldcs(reinterpret_cast<const uint4*>(src + (size_t)(2 * i) * kD));
    } else {
#pragma unroll
        for (int i = 0; i < kDecB16Rows; ++i) s[i] = make_uint4(0u, 0u, 0u, 0u);
    }

    for (int64_t t = 0; t < p.T; ++t) {
        const size_t tok = (size_t)n * p.T + t;
        const size_t row = tok * p.H + hm.hs;
        s_k[tid] = __bfloat162float(p.k[(tok * Hk + hm.hk) * kD + tid]);
        s_q[tid] = __bfloat162float(p.q[(tok * Hq + hm.hq) * kD + tid]);
        s_v[tid] = __bfloat162float(p.v[row * kD + tid]);
        s_e[tid] = expf(p.g[row * kD + tid]);
        const float beta_t = __bfloat162float(p.beta[row]);
        __syncthreads();

        // Pass 1: u = S'^T k and w = S'^T q over this thread's rows (S' = Diag(e) S).
        float u[8], w[8], qk = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) u[c] = w[c] = 0.f;
#pragma unroll
        for (int i = 0; i < kDecB16Rows; ++i) {
            const int r = rbase + 2 * i;
            const float er = s_e[r], kr = s_k[r], qr = s_q[r];
            qk = fmaf(qr, kr, qk);
            float x[8];
            unpack8(s[i], x);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float y = er * x[c];
                u[c] = fmaf(kr, y, u[c]);
                w[c] = fmaf(qr, y, w[c]);
            }
        }
        // The two half-warps hold the even and odd rows of the same columns.
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            u[c] += __shfl_xor_sync(0xffffffffu, u[c], 16);
            w[c] += __shfl_xor_sync(0xffffffffu, w[c], 16);
        }
        qk += __shfl_xor_sync(0xffffffffu, qk, 16);
        if (hw == 0) {
            float4* ru = reinterpret_cast<float4*>(&s_red[0][warp][c0]);
            float4* rw = reinterpret_cast<float4*>(&s_red[1][warp][c0]);
            ru[0] = make_float4(u[0], u[1], u[2], u[3]);
            ru[1] = make_float4(u[4], u[5], u[6], u[7]);
            rw[0] = make_float4(w[0], w[1], w[2], w[3]);
            rw[1] = make_float4(w[4], w[5], w[6], w[7]);
        }
        if (lane == 0) s_qk[warp] = qk;
        __syncthreads();

        // Column j = tid: delta_j and the output o_j.
        {
            float uu = 0.f, ww = 0.f, qq = 0.f;
#pragma unroll
            for (int x = 0; x < kDecB16Threads / 32; ++x) {
                uu += s_red[0][x][tid];
                ww += s_red[1][x][tid];
                qq += s_qk[x];
            }
            const float d = beta_t * (s_v[tid] - uu);
            s_d[tid] = d;
            p.out[(tok * Ho + ho) * kD + tid] = __float2bfloat16_rn(p.scale * fmaf(qq, d, ww));
        }
        __syncthreads();

        // Pass 2: S = Diag(e) S + k delta^T, rounded to bf16.
        float d[8];
        {
            const float4 a = *reinterpret_cast<const float4*>(&s_d[c0]);
            const float4 b = *reinterpret_cast<const float4*>(&s_d[c0 + 4]);
            d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
            d[4] = b.x; d[5] = b.y; d[6] = b.z; d[7] = b.w;
        }
#pragma unroll
        for (int i = 0; i < kDecB16Rows; ++i) {
            const int r = rbase + 2 * i;
            const float er = s_e[r], kr = s_k[r];
            float x[8];
            unpack8(s[i], x);
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = fmaf(kr, d[c], er * x[c]);
            s[i] = make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]),
                              pack2(x[6], x[7]));
        }
        // The next token overwrites the staged rows only after every warp has passed here.
        if (t + 1 < p.T) __syncthreads();
    }

    if (p.sfin && hm.state_owner) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.sfin) + soff;
#pragma unroll
        for (int i = 0; i < kDecB16Rows; ++i)
            __stcs(reinterpret_cast<uint4*>(dst + (size_t)(2 * i) * kD), s[i]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.N * (p.Hq > p.H ? p.Hq : p.H);
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)rows);
    const bool grouped = p.Hq != p.H;
    if (p.state_bf16) {
        if (grouped)
            kda_decode_bf16_kernel<true><<<grid, dim3(kDecB16Threads), 0, stream>>>(p);
        else
            kda_decode_bf16_kernel<false><<<grid, dim3(kDecB16Threads), 0, stream>>>(p);
    } else {
        if (grouped)
            kda_decode_kernel<true><<<grid, dim3(kDecThreads), 0, stream>>>(p);
        else
            kda_decode_kernel<false><<<grid, dim3(kDecThreads), 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
