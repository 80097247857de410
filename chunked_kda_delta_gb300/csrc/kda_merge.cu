// kda_merge.cu -- the "merge" step of segment-parallel prefill: the serial combine of
// per-segment summaries into the carry (state at each segment start).
//
// Segment pipeline (cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP
// prefill", commit notes: "Split long sequences into segments and run the recurrence per
// segment: K1 once -> pre_scan -> merge -> segment-K2").  Over one segment the state map
// is affine, S_end = m_seg S_start + b_seg, so
//     carry_0 = S_0 (or 0),   carry_{s+1} = m_seg[s] carry_s + b_seg[s].
// One CTA per (sequence, head, 32-column block of the carry): the carry's columns are
// independent, so each CTA runs the whole serial chain over segments for its block.
// fp32 throughout (the carries feed every later output of their segment).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kCols = 32;             // carry columns per CTA
constexpr int kMRow = kD + 4;         // padded row of the transposed transition in smem
constexpr int kCRow = kCols + 4;      // padded row of the carry block
constexpr int kMergeSmem = (kD * kMRow + kD * kCRow) * 4;

__global__ void __launch_bounds__(256)
kda_merge_kernel(const float* __restrict__ m_seg, const float* __restrict__ b_seg,
                 const float* __restrict__ s0, float* __restrict__ carries, int B, int nseg,
                 int H, const int32_t* __restrict__ seg_start) {
    extern __shared__ __align__(16) float sm[];
    float* Mt = sm;                  // Mt[k][i] = m[i][k]
    float* Cb = sm + kD * kMRow;     // carry block [k][c]
    const int tid = threadIdx.x;
    const int cb = blockIdx.x % (kD / kCols);
    const int h = (blockIdx.x / (kD / kCols)) % H;
    const int b = blockIdx.x / ((kD / kCols) * H);
    const int i0 = (tid >> 3) * 4;   // 4 rows
    const int c0 = (tid & 7) * 4;    // 4 columns of the block
    const size_t st = (size_t)kD * kD;
    // Dense: summaries [B][nseg-1][H], carries [B][nseg][H].  Varlen: every table indexed
    // by the global segment row g = seg_start[b] + s, sequence b owning its own count.
    size_t g0 = 0;
    int ns = nseg;
    if (seg_start) {
        g0 = (size_t)seg_start[b];
        ns = seg_start[b + 1] - seg_start[b];
    }
    auto carry_at = [&](int s) {
        return carries + ((seg_start ? g0 + s : (size_t)b * nseg + s) * H + h) * st;
    };
    auto summary_at = [&](const float* base, int s) {
        return base + ((seg_start ? g0 + s : (size_t)b * (nseg - 1) + s) * H + h) * st;
    };

    // carry_0
    for (int e = tid; e < kD * kCols; e += 256) {
        const int k = e / kCols, c = e % kCols;
        const float v = s0 ? s0[((size_t)b * H + h) * st + (size_t)k * kD + cb * kCols + c] : 0.f;
        Cb[k * kCRow + c] = v;
        carry_at(0)[(size_t)k * kD + cb * kCols + c] = v;
    }
    for (int s = 0; s + 1 < ns; ++s) {
        const float* M = summary_at(m_seg, s);
        const float* Bs = summary_at(b_seg, s);
        for (int e = tid; e < kD * kD; e += 256) {
            const int i = e / kD, k = e % kD;
            Mt[k * kMRow + i] = M[e];
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[a][c] = Bs[(size_t)(i0 + a) * kD + cb * kCols + c0 + c];
#pragma unroll 4
        for (int k = 0; k < kD; ++k) {
            const float4 mv = *reinterpret_cast<const float4*>(Mt + k * kMRow + i0);
            const float4 cv = *reinterpret_cast<const float4*>(Cb + k * kCRow + c0);
            const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
            const float cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(mm[a], cc[c], acc[a][c]);
        }
        __syncthreads();
        float* out = carry_at(s + 1);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            *reinterpret_cast<float4*>(Cb + (i0 + a) * kCRow + c0) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
            *reinterpret_cast<float4*>(out + (size_t)(i0 + a) * kD + cb * kCols + c0) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
        __syncthreads();
    }
}

}  // namespace

size_t merge_smem_bytes() { return kMergeSmem; }
const void* merge_kernel_symbol() { return reinterpret_cast<const void*>(&kda_merge_kernel); }

cudaError_t launch_merge(const float* m_seg, const float* b_seg, const float* s0, float* carries,
                         int32_t B, int32_t nseg, int32_t H, cudaStream_t stream,
                         const int32_t* seg_start) {
    const long long blocks = (long long)B * H * (kD / kCols);
    if (blocks == 0) return cudaSuccess;
    kda_merge_kernel<<<(unsigned)blocks, 256, kMergeSmem, stream>>>(m_seg, b_seg, s0, carries, B,
                                                                   nseg, H, seg_start);
    return cudaGetLastError();
}

// One CTA: validate cu_seqlens (cu[0] = 0, non-decreasing, cu[N] <= T_total), then an
// exclusive scan of max(1, ceil(len / seg_len)).  On malformed input the status word is
// set and the table is all zeros, so every segment row of the following launches exits.
__global__ void __launch_bounds__(1024)
kda_segment_table_kernel(const int32_t* __restrict__ cu, int N, long long T_total, long long seg_len,
                         int32_t* __restrict__ seg_start, int32_t* status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        bad = 0;
    }
    __syncthreads();
    for (int n = tid; n < N; n += blockDim.x) {
        const long long a = cu[n], e = cu[n + 1];
        if ((n == 0 && a != 0) || a < 0 || e < a || e > T_total) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicCAS(status, kStatusOk, kStatusBadSeqlens);
        for (int n = tid; n <= N; n += blockDim.x) seg_start[n] = 0;
        return;
    }
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int32_t cnt = 0;
        if (n < N) {
            const long long len = (long long)cu[n + 1] - cu[n];
            const long long c = (len + seg_len - 1) / seg_len;
            cnt = (int32_t)(c > 1 ? c : 1);
        }
        int32_t incl = cnt;  // inclusive warp scan
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += o;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t before = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - cnt;
        if (n < N) seg_start[n] = before;
        __syncthreads();
        if (tid == 0) carry += warp_sums[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) seg_start[N] = carry;
}

cudaError_t launch_segment_table(const int32_t* cu, int32_t N, int64_t T_total, int64_t seg_len,
                                 int32_t* seg_start, int32_t* status, cudaStream_t stream) {
    kda_segment_table_kernel<<<1, 1024, 0, stream>>>(cu, N, (long long)T_total, (long long)seg_len,
                                                    seg_start, status);
    return cudaGetLastError();
}

}  // namespace kda
