// kda_fwd_serial.cu -- fused K1 + K2 forward prefill, one CTA per (sequence, head).
//
// Chunkwise form of the KDA recurrence (CHUNK = 16, D = 128; cuLA PR #103
// "feat(kda/sm90): FlashKDA prefill port + intracard-CP prefill", commit notes:
// "K1 prepares decayed q/k, beta and the WY inverse; K2 runs the inter-chunk
// recurrence").  For a chunk of C rows with chunk-start state S (Dk x Dv):
//   gam_r  = sum_{m<=r} g_m                               (per channel)
//   A      = strict_lower(beta_r (k_r . k_s exp(gam_r - gam_s)))
//   W      = (I + A)^{-1} diag(beta) (K o exp(gam)),   U = (I + A)^{-1} diag(beta) V
//   delta  = U - W S
//   O      = scale (Qtil S + Mq delta),   Mq = lower(q_r . k_s exp(gam_r - gam_s))
//   S     <- Diag(exp gam_C) S + Kbar^T delta,   Kbar_r = k_r o exp(gam_C - gam_r)
// The pairwise decay exp(gam_r - gam_s) is factored through a reference row of
// the chunk (row 7): exp(gam_r - gam_ref) * exp(gam_ref - gam_s), so no factor
// leaves the fp32 range while the in-chunk log-decay span of a half chunk stays
// below ~80 per channel.
//
// This first kernel keeps everything in fp32 on the CUDA cores: the state lives
// in shared memory, each of the 256 threads owns value columns.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kRef = 7;

struct SimpleSmem {
    float S[kD * kD];         // state, [i_k][j_v]
    float Qt[kChunk * kD];    // q o exp(gam)
    float Wb[kChunk * kD];    // beta k o exp(gam) -> solved in place into W
    float Kbar[kChunk * kD];  // k o exp(gam_C - gam)
    float KQ[kChunk * kD];    // k o exp(gam - gam_ref)
    float QQ[kChunk * kD];    // q o exp(gam - gam_ref)
    float KK[kChunk * kD];    // k o exp(gam_ref - gam)
    float Ub[kChunk * kD];    // beta v -> solved in place into U
    float Dl[kChunk * kD];    // delta
    float A[kChunk * kChunk];
    float Mq[kChunk * kChunk];
    float GC[kD];             // exp(gam_C)
    float bet[kChunk];
};

__global__ void __launch_bounds__(kThreads, 1) kda_fwd_simple_kernel(FwdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimpleSmem& sm = *reinterpret_cast<SimpleSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int h = blockIdx.x % p.H;
    const int n = blockIdx.x / p.H;
    int64_t bos, eos;
    if (!seq_range(p, n, bos, eos)) return;
    const int64_t H = p.H;
    const size_t state_off = ((size_t)n * p.H + h) * kD * kD;

    for (int e = tid; e < kD * kD; e += kThreads)
        sm.S[e] = p.s0 ? p.s0[state_off + e] : 0.f;
    __syncthreads();

    for (int64_t t0 = bos; t0 < eos; t0 += kChunk) {
        const int C = (eos - t0 < kChunk) ? (int)(eos - t0) : kChunk;
        if (tid < kChunk)
            sm.bet[tid] = tid < C ? __bfloat162float(p.beta[(t0 + tid) * H + h]) : 0.f;
        __syncthreads();

        if (tid < kD) {
            // K1: cumulative gate and the decayed operands for channel c.
            const int c = tid;
            float gm[kChunk];
            float acc = 0.f;
#pragma unroll
            for (int r = 0; r < kChunk; ++r) {
                acc += r < C ? p.g[((t0 + r) * H + h) * kD + c] : 0.f;
                gm[r] = acc;
            }
            const float gref = gm[kRef], glast = gm[kChunk - 1];
            sm.GC[c] = __expf(glast);
#pragma unroll
            for (int r = 0; r < kChunk; ++r) {
                const size_t off = ((t0 + r) * H + h) * kD + c;
                const float kr = r < C ? __bfloat162float(p.k[off]) : 0.f;
                const float qr = r < C ? __bfloat162float(p.q[off]) : 0.f;
                const float e = __expf(gm[r]);
                sm.Qt[r * kD + c] = qr * e;
                sm.Wb[r * kD + c] = sm.bet[r] * kr * e;
                sm.Kbar[r * kD + c] = kr * __expf(glast - gm[r]);
                const float up = __expf(gm[r] - gref), dn = __expf(gref - gm[r]);
                sm.KQ[r * kD + c] = kr * up;
                sm.QQ[r * kD + c] = qr * up;
                sm.KK[r * kD + c] = kr * dn;
            }
        } else {
            const int j = tid - kD;
#pragma unroll
            for (int r = 0; r < kChunk; ++r) {
                const float vr = r < C ? __bfloat162float(p.v[((t0 + r) * H + h) * kD + j]) : 0.f;
                sm.Ub[r * kD + j] = sm.bet[r] * vr;
            }
        }
        __syncthreads();

        {   // K1: in-chunk Grams, one (r, s) pair per thread.
            const int r = tid >> 4, s = tid & 15;
            float a = 0.f, m = 0.f;
            if (s <= r) {
#pragma unroll 8
                for (int c = 0; c < kD; ++c) {
                    const float ks = sm.KK[s * kD + c];
                    a = fmaf(sm.KQ[r * kD + c], ks, a);
                    m = fmaf(sm.QQ[r * kD + c], ks, m);
                }
            }
            sm.A[r * kChunk + s] = s < r ? sm.bet[r] * a : 0.f;
            sm.Mq[r * kChunk + s] = s <= r ? m : 0.f;
        }
        __syncthreads();

        {   // K1: WY solve (I + A) X = rhs, forward substitution, one column per thread.
            float* X = tid < kD ? sm.Wb : sm.Ub;
            const int col = tid & (kD - 1);
            float x[kChunk];
#pragma unroll
            for (int r = 0; r < kChunk; ++r) {
                float acc = X[r * kD + col];
#pragma unroll
                for (int s = 0; s < r; ++s) acc = fmaf(-sm.A[r * kChunk + s], x[s], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < kChunk; ++r) X[r * kD + col] = x[r];
        }
        __syncthreads();

        // K2: delta = U - W S and the Qtil S part of the output.
        const int j = tid & (kD - 1);
        const int r0 = tid >> 7;
        float accd[8], acco[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) accd[m] = acco[m] = 0.f;
        for (int i = 0; i < kD; ++i) {
            const float sij = sm.S[i * kD + j];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = r0 + 2 * m;
                accd[m] = fmaf(sm.Wb[r * kD + i], sij, accd[m]);
                acco[m] = fmaf(sm.Qt[r * kD + i], sij, acco[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int r = r0 + 2 * m;
            sm.Dl[r * kD + j] = sm.Ub[r * kD + j] - accd[m];
        }
        __syncthreads();

        // K2: output rows and the state update.
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int r = r0 + 2 * m;
            float o = acco[m];
            for (int s = 0; s <= r; ++s) o = fmaf(sm.Mq[r * kChunk + s], sm.Dl[s * kD + j], o);
            if (r < C) p.out[((t0 + r) * H + h) * kD + j] = __float2bfloat16_rn(p.scale * o);
        }
        for (int i = r0; i < kD; i += 2) {
            float acc = sm.GC[i] * sm.S[i * kD + j];
#pragma unroll
            for (int r = 0; r < kChunk; ++r) acc = fmaf(sm.Kbar[r * kD + i], sm.Dl[r * kD + j], acc);
            sm.S[i * kD + j] = acc;
        }
        __syncthreads();
    }

    if (p.sfin)
        for (int e = tid; e < kD * kD; e += kThreads) p.sfin[state_off + e] = sm.S[e];
}

}  // namespace

size_t serial_smem_bytes() { return sizeof(SimpleSmem); }
const void* serial_kernel_symbol() { return reinterpret_cast<const void*>(&kda_fwd_simple_kernel); }

cudaError_t launch_serial(const FwdParams& p, cudaStream_t stream) {
    const long long blocks = (long long)p.N * p.H;
    if (blocks == 0) return cudaSuccess;
    kda_fwd_simple_kernel<<<(unsigned)blocks, kThreads, sizeof(SimpleSmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
